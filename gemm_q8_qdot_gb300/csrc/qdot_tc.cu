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
// Q8_0 block is two K = 16 MMAs into a fresh TMEM accumulator.  (GB300's
// dense int8 tensor rate is far below its f16 rate, and ptxas does not take
// the integer MMA kind for sm_103a.)
//
// Scale products on the tensor core.  The per-block factor xs[p, b] * ys[q, b]
// is itself a rank-1 product, so a third MMA per block (bf16, K = 16) writes
// the 128 x BN tile of factors P next to S in TMEM: each f32 scale is split
// exactly into three bf16 (hi + mid + lo, each the rounded remainder of the
// previous), and the K = 16 operand rows [h h h m m m l l l 0 ..] of X and
// [h m l h m l h m l 0 ..] of Y multiply out to all nine cross terms, whose
// f32 sum is xs * ys up to f32 rounding.  The epilogue is then one tcgen05.ld
// of S, one of P and one FFMA per output per block: acc += P * S.
//
// Tile.  The "P" operand X (128 rows per tile, the MMA M and the TMEM lanes)
// and the "Q" operand Y (BN rows, the MMA N) are both K-major int8 [rows, K].
// For M > 64, X = A and Y = W (output C[p * N + q], BN = 128); for M <= 64,
// X = W and Y = A with BN = M rounded up to 16, 32 or 64 (output C[q * N + p]),
// so that the large weight matrix fills the 128-row side.
//
// Work.  Persistent CTAs (at most one per SM) take (P tile, Q tile, K split)
// units round-robin, the P tile varying fastest.  K is split only when the
// tiles are too few to spread evenly over the SMs; split units add their
// partial sums into a zeroed C with atomics.
//
// Pipeline (warp-specialised, all hand-offs through mbarriers):
//   warp 0      TMA producer: per int8 stage (one scale group of 4 blocks,
//               128 K) a 128-byte-swizzled int8 box of X and of Y and the
//               two f32 scale boxes, on one barrier (int8 ring, S8 deep);
//   warps 2..7  converters: int8 -> f16 (the byte b is biased to b + 128,
//               placed under the f16 exponent of 1024 and 1152 subtracted,
//               all exact) into the UMMA K-major 128-byte-swizzle layout, two
//               f16 stages of 64 K per int8 stage, plus the bf16 split
//               operands of the stage's scale products (f16 ring, S16 deep);
//   warp 1      MMA issuer (one thread): 2 S-MMAs + 1 P-MMA per block into
//               one of NBUF TMEM buffer pairs, tcgen05.commit -> tfull;
//               commits also free the f16 stages;
//   warps 8..15 epilogue: four TMEM lane quadrants x two column halves;
//               acc += P * S in registers; the unit's last block stores C
//               (float4 when the rows are 16-byte aligned).
//
// Safety.  Every mbarrier wait is bounded (a clock64 limit).  A wait that
// gives up sets the library's device status word and a CTA-wide abort flag;
// every role then runs out its loops without waiting or working (so no
// barrier is skipped), TMA loads and MMAs still in flight are drained with
// bounded waits, TMEM is freed and the kernel returns.  The host reads the
// status with pq_check_device.  No trap, no unbounded spin.
#include <cuda.h>
#include <cuda_bf16.h>
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

constexpr int BM = 128;      // rows of the MMA's A operand per tile (MMA M, TMEM lanes)
constexpr int KS = 64;       // K elements per f16 stage (two Q8_0 blocks)
constexpr int KS8 = 128;     // K elements per int8 stage (one scale group): 128-byte TMA rows
constexpr int GROUP = 4;     // Q8_0 blocks per scale group (128 K, two stages)
// One f16 stage of the pre-tiled X operand (PREX): the 128 x 64 f16 tile in
// the UMMA K-major 128-byte-swizzle layout, then the scale-product operands of
// its two Q8_0 blocks (128 rows x 16 bf16 each, K-major without swizzle).
constexpr int kXtF16 = BM * KS * 2;
constexpr int kXtStage = kXtF16 + 2 * BM * 32;
// Q5_0 weight blocks ("Phobos Language Spec" section 10, Q5_0 row): 20 bytes per
// 32 elements, the qh word then 16 bytes whose byte e holds element e in its low
// nibble and element e + 16 in its high nibble, each element q - 16.  One scale
// group (4 blocks, 128 K) of a row is 80 bytes.
constexpr int kQ5Block = 20;
constexpr int kQ5Row = GROUP * kQ5Block;

struct TcParams {
    const float* xs;          // scale of MMA-A row p, block b: xs[p * xs_r + b * xs_b]
    int64_t xs_r, xs_b;
    const float* ys;          // scale of MMA-B row q, block b: ys[q * ys_r + b * ys_b]
    int64_t ys_r, ys_b;
    float* C;                 // C[p * ldp + q * ldq]
    int64_t ldp, ldq;
    int32_t* S;               // block sums (verification): S[p * sp + q * sq + b]
    int64_t sp, sq;
    int64_t P, Q, K;
    int groups_per_split;
    int splits;               // K splits per tile
    int tiles_p;              // tiles along P
    int units;                // tiles_p * tiles_q * splits work units, taken round-robin by the CTAs
    int atomic;               // split-K: red.add into a zeroed C
    int vec_store;            // ldq == 1, Q % 4 == 0, C 16-byte aligned: float4 stores
    int has_scales;           // 0 in block-sum mode (no scale planes)
    int xs_sr, xs_sb;         // scale tile in shared memory: xs(row, blk) at row * xs_sr + blk * xs_sb
    int ys_sr, ys_sb;
    int inject_skip_stage;    // test hook: the producer skips this stage (-1: off)
    unsigned long long timeout_cycles;
    int regsplit;             // 1: move registers from the producer / converter warps to the epilogue
    const uint8_t* xt;        // pre-tiled X (PREX kernels): kXtStage bytes per (P tile, f16 stage)
    int64_t xt_tile_stride;   // bytes per P tile of xt
};

// MMA-A ("X", 128 rows per tile) and MMA-B ("Y", BN rows) both arrive as int8
// by TMA into the int8 ring and are converted to f16 by the converter warps.
// The f32 scales of the stage's 4 blocks arrive by TMA with the int8 tiles;
// the converters turn them into the scale-product MMA's operands (exact 3-way
// bf16 splits) in the f16 stage.
//
// ESC (narrow tiles): no scale-product MMA.  A TMEM buffer holds the block sums
// of one scale group (4 blocks x BN columns) and the epilogue multiplies them by
// the two f32 scales, read from the group's int8 stage, which it releases.
template <int BN, int NCONV, int NEPI, int S8, int S16, bool Q5 = false, bool ESC = false>
struct Cfg {
    static constexpr int kThreads = 32 * (2 + NCONV + NEPI);
    static constexpr int kE0 = 2 + NCONV;                 // first epilogue warp
    static constexpr int kBufCols = ESC ? GROUP * BN : 2 * BN;  // TMEM columns per buffer
    static constexpr int kNbufMax = ESC ? 3 : 4;
    static constexpr int kNbuf = (512 / kBufCols) < kNbufMax ? (512 / kBufCols) : kNbufMax;  // TMEM buffers
    static constexpr int kTmemUsed = kNbuf * kBufCols;
    static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                     : kTmemUsed <= 256 ? 256 : 512;
    static constexpr int kCW = BN / (NEPI / 4);          // columns per epilogue warp
    static constexpr int kCH = kCW < (ESC ? 8 : 16) ? kCW : (ESC ? 8 : 16);  // columns per tcgen05.ld
    static constexpr int kX8 = BM * KS8;                  // int8 X tile bytes (one TMA box)
    static constexpr int kY8 = BN * (Q5 ? kQ5Row : KS8);  // Y tile of one scale group (int8 or Q5_0 blocks)
    static constexpr int kXS = BM * GROUP * 4;            // f32 scales of the stage's 4 blocks
    static constexpr int kYS = BN * GROUP * 4;
    static constexpr int kX16 = BM * KS * 2;              // f16 X tile bytes
    static constexpr int kY16 = BN * KS * 2;
    static constexpr int kXP = ESC ? 0 : BM * 32;         // scale-product operand, one block: [rows][16] bf16
    static constexpr int kYP = ESC ? 0 : BN * 32;
    static constexpr int kOffX8 = 0;
    static constexpr int kOffY8 = kOffX8 + S8 * kX8;
    static constexpr int kOffX16 = kOffY8 + S8 * kY8;
    static constexpr int kOffY16 = kOffX16 + S16 * kX16;
    static constexpr int kOffXP = kOffY16 + S16 * kY16;   // S16 x 2 blocks
    static constexpr int kOffYP = kOffXP + S16 * 2 * kXP;
    static constexpr int kOffXS = kOffYP + S16 * 2 * kYP;  // S8 x scale tiles, with the int8 stages
    static constexpr int kOffYS = kOffXS + S8 * kXS;
    static constexpr int kOffBar = kOffYS + S8 * kYS;
    static constexpr int kNumBars = 2 * S8 + 2 * S16 + 2 * kNbuf + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmem = kOffMisc + 16 + 1024;    // + alignment slack
    static constexpr int kOct = (BM + BN) / 8;            // row octets converted per f16 stage
    static constexpr int kSplitPerThread = ((BM + BN) * 2 + NCONV * 32 - 1) / (NCONV * 32);
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
    static_assert(NEPI == 8, "epilogue warps: two column halves over the four TMEM lane quadrants");
    static_assert(kCW % kCH == 0 && kCH % 8 == 0, "epilogue column chunks");
    static_assert(kX8 % 1024 == 0 && kY8 % 1024 == 0 && kX16 % 1024 == 0 && kY16 % 1024 == 0, "1024-B tiles");
    static_assert(!Q5 || BN % 8 == 0, "Q5_0 weights: whole row octets");
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(!ESC || !Q5, "scales in the epilogue: Q8_0 weights only");
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
    for (uint32_t n = 1;; ++n) {
        if (tc::mbar_try_wait(bar, parity)) return true;
        if ((n & 31) == 0) {
            if (*abort_flag) return false;
            if (static_cast<unsigned long long>(clock64() - t0) > limit) {
                set_abort(abort_flag);
                return false;
            }
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

// Q5_0: the four bits of x spread to bit 0 of four bytes (x * 0x00204081 puts
// bit i at bit 8i, no carries), and four biased elements q in [0, 31] (one per
// byte) -> two f16x2 of q - 16, exact (placed under the f16 exponent of 1024,
// 1040 = 1024 + 16 subtracted).
__device__ __forceinline__ uint32_t q5_spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

__device__ __forceinline__ void q5_to_f16x4(uint32_t q, uint32_t& lo, uint32_t& hi) {
    const uint32_t a = __byte_perm(q, 0x64646464u, 0x4140u);
    const uint32_t b = __byte_perm(q, 0x64646464u, 0x4342u);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6410u), __ushort_as_half(0x6410u));
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
}

// Exact split of an f32 into three bf16 whose sum is the value (normal range).
__device__ __forceinline__ void split3_bf16(float x, uint32_t& h, uint32_t& m, uint32_t& l) {
    const __nv_bfloat16 bh = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(bh);
    const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(bm);
    const __nv_bfloat16 bl = __float2bfloat16_rn(r2);
    h = __bfloat16_as_ushort(bh);
    m = __bfloat16_as_ushort(bm);
    l = __bfloat16_as_ushort(bl);
}

template <int BN, int NCONV, int NEPI, int S8, int S16, int MINB, bool SUMS, bool PREX, bool Q5, bool ESC>
__global__ void __launch_bounds__(Cfg<BN, NCONV, NEPI, S8, S16, Q5, ESC>::kThreads, MINB)
qdot_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
               const __grid_constant__ CUtensorMap tmXS, const __grid_constant__ CUtensorMap tmYS,
               const TcParams prm) {
    using CF = Cfg<BN, NCONV, NEPI, S8, S16, Q5, ESC>;
    static_assert(!ESC || (!SUMS && !PREX), "scales in the epilogue: scaled output, in-kernel X");
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
    const uint32_t sbase = tc::smem_u32(smem);  // the same bytes in the shared window

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = prm.timeout_cycles;

    const int ngroups = static_cast<int>(prm.K / (KS * 2));
    // work unit u -> (tile along P, tile along Q, K split); stages of the unit
    struct Unit {
        int64_t p0, q0;
        int g_begin, nst;
    };
    auto unit = [&](int u) {
        Unit r;
        // the P tile varies fastest: CTAs running at the same time share Q tiles
        // (the operand with more tiles) and spread their reads of the P operand
        const int z = u % prm.splits;
        const int t = u / prm.splits;
        r.p0 = static_cast<int64_t>(t % prm.tiles_p) * BM;
        r.q0 = static_cast<int64_t>(t / prm.tiles_p) * BN;
        r.g_begin = z * prm.groups_per_split;
        r.nst = 2 * max(0, min(ngroups, r.g_begin + prm.groups_per_split) - r.g_begin);
        return r;
    };
    // The CTA's units: round-robin for the 128-column tiles (the prompt shapes:
    // CTAs running at the same time then share weight tiles in L2); a
    // contiguous range for the narrow tiles, whose K is split, so that a tile's
    // consecutive splits run on one CTA, which adds them in registers and
    // writes the tile once.
    const int u_first = ESC ? static_cast<int>(static_cast<int64_t>(blockIdx.x) * prm.units / gridDim.x)
                            : static_cast<int>(blockIdx.x);
    const int u_end = ESC ? static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * prm.units / gridDim.x)
                          : prm.units;
    const int u_step = ESC ? 1 : static_cast<int>(gridDim.x);

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S8; ++i) {
            tc::mbar_init(&full8[i], 1);
            tc::mbar_init(&empty8[i], NCONV + (ESC ? NEPI : 0));  // ESC: + the epilogue's reads of the scales
        }
        for (int i = 0; i < S16; ++i) {
            tc::mbar_init(&full16[i], NCONV + (PREX ? 1 : 0));  // + the producer's copy of pre-tiled X
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
        if (prm.has_scales) {
            tc::tma_prefetch_map(&tmXS);
            tc::tma_prefetch_map(&tmYS);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, CF::kTmemCols);
        tc::tmem_relinquish();
        tc::tc_fence_before_sync();
    }
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Register split between the roles.  The launch gives each of the 512 threads
    // 128 registers; the warpgroups of the producer, the MMA issuer and the
    // converters (warps 0-7) give 16 each to the epilogue warpgroups (warps 8-15),
    // whose 64 accumulators and TMEM chunks then fit without spilling:
    // 256 x 112 + 256 x 144 = 65,536 = the launch's total.  The host sets regsplit
    // only after checking that the kernel was built with exactly 128 registers.
    if constexpr (CF::kThreads == 512 && CF::kE0 == 8) {
        if (prm.regsplit) {
            if (warp < CF::kE0) asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
            else asm volatile("setmaxnreg.inc.sync.aligned.u32 144;" ::: "memory");
        }
    }
    // everything below reads global memory the preceding kernel may have written
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // One int8 stage = one scale group = 128 K = two f16 stages: the int8
        // tiles of X and Y and their f32 scales, four TMA boxes on one barrier.
        // With pre-tiled X (PREX) the int8 stage holds Y and its scales only, and
        // each f16 stage's X tile and X scale-product operands arrive by one bulk
        // copy straight into the f16 ring (the converters then handle Y alone).
        if (lane == 0) {
            const uint32_t tx = (PREX ? 0 : CF::kX8) + CF::kY8 +
                                (prm.has_scales ? (PREX ? 0 : CF::kXS) + CF::kYS : 0);
            int issued8 = 0, issued16 = 0;
            int gi = 0;  // int8-stage counter over all units of this CTA
            for (int u = u_first; u < u_end; u += u_step) {
                const Unit un = unit(u);
                const int n8 = un.nst / 2;
                for (int i = 0; i < n8; ++i, ++gi) {
                    const int s8 = gi % S8;
                    const int g = un.g_begin + i;  // scale group = int8 stage along K
                    if (!bounded_wait(&empty8[s8], ((gi / S8) & 1) ^ 1, abort_flag, limit)) continue;
                    issued8 = gi + 1;
                    if (gi != prm.inject_skip_stage) {  // test hook: the skipped stage never arrives
                        tc::mbar_arrive_expect_tx(&full8[s8], tx);
                        if (!PREX)
                            tc::tma_load_2d(smem + CF::kOffX8 + s8 * CF::kX8, &tmX, &full8[s8], g * KS8,
                                            static_cast<int>(un.p0));
                        tc::tma_load_2d(smem + CF::kOffY8 + s8 * CF::kY8, &tmY, &full8[s8], g * (Q5 ? kQ5Row : KS8),
                                        static_cast<int>(un.q0));
                        if (prm.has_scales) {
                            // row-major planes: box {4 blocks, rows}; block-major: box {rows, 4 blocks}
                            const int b0 = g * GROUP;
                            if (!PREX)
                                tc::tma_load_2d(smem + CF::kOffXS + s8 * CF::kXS, &tmXS, &full8[s8],
                                                prm.xs_sb == 1 ? b0 : static_cast<int>(un.p0),
                                                prm.xs_sb == 1 ? static_cast<int>(un.p0) : b0);
                            tc::tma_load_2d(smem + CF::kOffYS + s8 * CF::kYS, &tmYS, &full8[s8],
                                            prm.ys_sb == 1 ? b0 : static_cast<int>(un.q0),
                                            prm.ys_sb == 1 ? static_cast<int>(un.q0) : b0);
                        }
                    }
                    if constexpr (PREX) {
#pragma unroll 1
                        for (int h = 0; h < 2; ++h) {
                            const int gi16 = gi * 2 + h;
                            const int s16 = gi16 % S16;
                            if (!bounded_wait(&empty16[s16], ((gi16 / S16) & 1) ^ 1, abort_flag, limit)) continue;
                            issued16 = gi16 + 1;
                            const uint8_t* src = prm.xt + (un.p0 / BM) * prm.xt_tile_stride +
                                                 static_cast<int64_t>(g * 2 + h) * kXtStage;
                            tc::mbar_arrive_expect_tx(&full16[s16], kXtStage);
                            tc::bulk_copy_g2s(smem + CF::kOffX16 + s16 * CF::kX16, src, kXtF16, &full16[s16]);
                            tc::bulk_copy_g2s(smem + CF::kOffXP + s16 * 2 * CF::kXP, src + kXtF16, 2 * CF::kXP,
                                              &full16[s16]);
                        }
                    }
                }
            }
            // copies in flight land before the CTA may exit
            for (int i = max(0, issued8 - S8); i < issued8; ++i)
                if (i != prm.inject_skip_stage) drain_wait(&full8[i % S8], (i / S8) & 1, limit);
            if constexpr (PREX)
                for (int i = max(0, issued16 - S16); i < issued16; ++i) drain_wait(&full16[i % S16], (i / S16) & 1, limit);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(BM, BN);
            constexpr uint32_t idesc_p = tc::idesc_bf16_f32(BM, BN);
            int g = 0, gi = 0;  // g: TMEM hand-offs (blocks, or ESC scale groups)
            bool gok = false;   // ESC: the group's buffer was free
            for (int u = u_first; u < u_end; u += u_step) {
                const int nst = unit(u).nst;
                for (int i = 0; i < nst; ++i, ++gi) {
                    const int s = gi % S16;
                    const bool ok = bounded_wait(&full16[s], (gi / S16) & 1, abort_flag, limit);
                    if (ok) tc::tc_fence_after_sync();
                    const uint32_t xa = sbase + CF::kOffX16 + s * CF::kX16;
                    const uint32_t ya = sbase + CF::kOffY16 + s * CF::kY16;
                    if constexpr (ESC) {
                        // this f16 stage holds blocks 2h and 2h + 1 of the group (units start
                        // at group boundaries): their block sums go to columns (2h + bb) * BN
                        // of the group's buffer, handed to the epilogue after the second half
                        const int h = i & 1;
                        const int buf = g % CF::kNbuf;
                        if (h == 0) gok = ok && bounded_wait(&tempty[buf], ((g / CF::kNbuf) & 1) ^ 1, abort_flag, limit);
                        if (ok && gok) {
                            tc::tc_fence_after_sync();
#pragma unroll
                            for (int bb = 0; bb < 2; ++bb) {
                                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * CF::kBufCols + (h * 2 + bb) * BN);
#pragma unroll
                                for (int kk = 0; kk < 2; ++kk) {
                                    const uint32_t koff = static_cast<uint32_t>((bb * 2 + kk) * 32);
                                    tc::umma_f16(d, tc::sw128_kmajor_desc(xa + koff), tc::sw128_kmajor_desc(ya + koff),
                                                 idesc, kk);
                                }
                            }
                        }
                        if (h == 1) {
                            if (gok) tc::umma_commit(&tfull[buf]);
                            ++g;
                        }
                    } else {
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb, ++g) {
                            const int buf = g % CF::kNbuf;
                            if (!ok || !bounded_wait(&tempty[buf], ((g / CF::kNbuf) & 1) ^ 1, abort_flag, limit))
                                continue;
                            tc::tc_fence_after_sync();
                            const uint32_t d = tmem_base + static_cast<uint32_t>(buf * 2 * BN);
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t koff = static_cast<uint32_t>((bb * 2 + kk) * 32);  // 16 f16 = 32 B
                                tc::umma_f16(d, tc::sw128_kmajor_desc(xa + koff), tc::sw128_kmajor_desc(ya + koff),
                                             idesc, kk);
                            }
                            // P = (split xs) . (split ys)^T: the scale products of this block
                            const uint32_t xp = sbase + CF::kOffXP + (s * 2 + bb) * CF::kXP;
                            const uint32_t yp = sbase + CF::kOffYP + (s * 2 + bb) * CF::kYP;
                            tc::umma_f16(d + BN, tc::noswz_kmajor_desc(xp, 128, 256), tc::noswz_kmajor_desc(yp, 128, 256),
                                         idesc_p, 0);
                            tc::umma_commit(&tfull[buf]);
                        }
                    }
                    // release the f16 stage once its MMAs completed
                    tc::umma_commit(&empty16[s]);
                }
            }
            tc::umma_commit(drain);  // arrives when every MMA issued above has completed
            drain_wait(drain, 0, limit);
        }
    } else if (warp < CF::kE0) {
        // ------------------------------------------------------------ converters
        // each int8 stage (128 K) becomes two f16 stages (64 K each)
        const int cw = warp - 2;
        const int ct = cw * 32 + lane;  // 0 .. 32 * NCONV - 1
        const int r_in = lane & 7;      // row within an octet
        const int c4 = lane >> 3;       // 16-byte chunk within this half's 64 bytes of an int8 row
        int g8 = 0, g16 = 0;
        for (int u = u_first; u < u_end; u += u_step) {
            const int n8 = unit(u).nst / 2;
            for (int i = 0; i < n8; ++i, ++g8) {
                const int s8 = g8 % S8;
                int ok8 = 0;
                if (lane == 0) ok8 = bounded_wait(&full8[s8], (g8 / S8) & 1, abort_flag, limit);
                ok8 = __shfl_sync(0xffffffffu, ok8, 0);
                const uint32_t x8 = sbase + CF::kOffX8 + s8 * CF::kX8;
                const uint32_t y8 = sbase + CF::kOffY8 + s8 * CF::kY8;
                const uint32_t xs8 = sbase + CF::kOffXS + s8 * CF::kXS;
                const uint32_t ys8 = sbase + CF::kOffYS + s8 * CF::kYS;
#pragma unroll 1
                for (int h = 0; h < 2; ++h, ++g16) {
                    const int s16 = g16 % S16;
                    int ok = 0;
                    if (lane == 0)
                        ok = ok8 && bounded_wait(&empty16[s16], ((g16 / S16) & 1) ^ 1, abort_flag, limit);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok) {
                        const uint32_t x16 = sbase + CF::kOffX16 + s16 * CF::kX16;
                        const uint32_t y16 = sbase + CF::kOffY16 + s16 * CF::kY16;
                        const int c8 = h * 4 + c4;  // 16-byte chunk of the 128-byte int8 row
                        // octets of int8 rows converted per warp (Y rows only with pre-tiled X;
                        // X rows only with Q5_0 weights, which are decoded below)
                        constexpr int kOctEnd = Q5 ? BM / 8 : CF::kOct;
                        constexpr int kOw = PREX ? (Q5 ? 0 : (BN / 8 + NCONV - 1) / NCONV)
                                                 : (kOctEnd + NCONV - 1) / NCONV;
                        uint4 v[kOw > 0 ? kOw : 1];
#pragma unroll
                        for (int t = 0; t < kOw; ++t) {  // all loads first
                            const int o = (PREX ? BM / 8 : 0) + cw + t * NCONV;
                            if (o < kOctEnd) {
                                const bool isx = o < BM / 8;
                                const int row = (isx ? o : o - BM / 8) * 8 + r_in;
                                v[t] = tc::lds128((isx ? x8 : y8) + row * KS8 + ((c8 ^ (row & 7)) << 4));
                            }
                        }
#pragma unroll
                        for (int t = 0; t < kOw; ++t) {
                            const int o = (PREX ? BM / 8 : 0) + cw + t * NCONV;
                            if (o < kOctEnd) {
                                const bool isx = o < BM / 8;
                                const int row = (isx ? o : o - BM / 8) * 8 + r_in;
                                uint4 o0, o1;
                                i8x4_to_f16x4(v[t].x, o0.x, o0.y);
                                i8x4_to_f16x4(v[t].y, o0.z, o0.w);
                                i8x4_to_f16x4(v[t].z, o1.x, o1.y);
                                i8x4_to_f16x4(v[t].w, o1.z, o1.w);
                                const uint32_t dst = (isx ? x16 : y16) + row * (KS * 2);
                                tc::sts128(dst + (((2 * c4) ^ (row & 7)) << 4), o0);
                                tc::sts128(dst + (((2 * c4 + 1) ^ (row & 7)) << 4), o1);
                            }
                        }
                        if constexpr (Q5) {
                            // Y = the Q5_0 weight: one (row, block) of this f16 stage per task; the
                            // 32 elements (q - 16) become four 16-byte f16 chunks of the row
                            constexpr int kTasks = (BN * 2 + NCONV * 32 - 1) / (NCONV * 32);
#pragma unroll
                            for (int t = 0; t < kTasks; ++t) {
                                const int w = ct + t * NCONV * 32;
                                if (w < BN * 2) {
                                    const int row = w >> 1, bb = w & 1;
                                    const uint32_t src = y8 + row * kQ5Row + (h * 2 + bb) * kQ5Block;
                                    const uint32_t qh = tc::lds32(src);
                                    uint32_t d[4];
#pragma unroll
                                    for (int i = 0; i < 4; ++i) d[i] = tc::lds32(src + 4 + 4 * i);
                                    const uint32_t dst = y16 + row * (KS * 2);
#pragma unroll
                                    for (int c = 0; c < 4; ++c) {
                                        // chunk c: elements 8c .. 8c + 7 = two words of biased bytes q in [0, 31]
                                        uint32_t u[2];
#pragma unroll
                                        for (int hw = 0; hw < 2; ++hw) {
                                            const int e0 = 8 * c + 4 * hw;  // first element of the word
                                            const int i = (e0 & 15) >> 2;   // data word holding it
                                            const uint32_t nib = e0 < 16 ? (d[i] & 0x0f0f0f0fu) : ((d[i] >> 4) & 0x0f0f0f0fu);
                                            u[hw] = nib | (q5_spread4((qh >> e0) & 0xfu) << 4);
                                        }
                                        uint4 o;
                                        q5_to_f16x4(u[0], o.x, o.y);
                                        q5_to_f16x4(u[1], o.z, o.w);
                                        tc::sts128(dst + (((bb * 4 + c) ^ (row & 7)) << 4), o);
                                    }
                                }
                            }
                        }
                        // scale-product operands of this f16 stage's two blocks: row r, block bb ->
                        // 16 bf16 [h h h m m m l l l 0..] (X) or [h m l h m l h m l 0..] (Y),
                        // K-major without swizzle: 8-row x 16-byte core matrices, the two
                        // K halves 128 B apart, 8-row groups 256 B apart
                        constexpr int kSp = ESC ? 0 : PREX ? (BN * 2 + NCONV * 32 - 1) / (NCONV * 32) : CF::kSplitPerThread;
#pragma unroll
                        for (int t = 0; t < kSp; ++t) {
                            const int w = ct + t * NCONV * 32;
                            constexpr int kRows = PREX ? BN : BM + BN;  // rows whose scales are split here
                            if (w < kRows * 2) {
                                const int bb = w / kRows;
                                const int r = (PREX ? BM : 0) + w - bb * kRows;
                                const int blk = h * 2 + bb;  // block within the scale group
                                const bool isx = r < BM;
                                const int row = isx ? r : r - BM;
                                const float sc = tc::lds32f(isx ? xs8 + (row * prm.xs_sr + blk * prm.xs_sb) * 4
                                                                : ys8 + (row * prm.ys_sr + blk * prm.ys_sb) * 4);
                                uint32_t sh, sm, sl3;
                                split3_bf16(sc, sh, sm, sl3);
                                uint4 k0;
                                if (isx)
                                    k0 = make_uint4(sh | (sh << 16), sh | (sm << 16), sm | (sm << 16), sl3 | (sl3 << 16));
                                else
                                    k0 = make_uint4(sh | (sm << 16), sl3 | (sh << 16), sm | (sl3 << 16), sh | (sm << 16));
                                const uint4 k1 = make_uint4(sl3, 0u, 0u, 0u);
                                const uint32_t base = sbase + (isx ? CF::kOffXP + (s16 * 2 + bb) * CF::kXP
                                                                   : CF::kOffYP + (s16 * 2 + bb) * CF::kYP);
                                const uint32_t a0 = base + (row >> 3) * 256 + (row & 7) * 16;
                                tc::sts128(a0, k0);
                                tc::sts128(a0 + 128, k1);
                            }
                        }
                        tc::fence_proxy_async_smem();
                    }
                    __syncwarp();
                    // arrive also after an abort: the producer's drain and every later wait
                    // then find the barriers in a consistent phase
                    if (lane == 0) tc::mbar_arrive(&full16[s16]);
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&empty8[s8]);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        constexpr int NCH = CF::kCW / CF::kCH;
        const int e = warp - CF::kE0;
        const int quad = warp & 3;
        const int cb = (e >> 2) * CF::kCW;
        const int prow = quad * 32 + lane;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);

        uint64_t acc[CF::kCW / 2];  // f32 pairs: columns cb + 2t, cb + 2t + 1
#pragma unroll
        for (int t = 0; t < CF::kCW / 2; ++t) acc[t] = 0ull;

        int g = 0;  // block counter over all units of this CTA
        for (int u = u_first; u < u_end; u += u_step) {
            const Unit cu = unit(u);
            const int nblk = cu.nst * 2;
            const int64_t p = cu.p0 + prow;
            const bool pv = p < prm.P;
            if constexpr (ESC) {
                // one hand-off per scale group: block sums S_b (b = 0..3) in columns b * BN of the
                // buffer; out += (xs[p, b] * ys[q, b]) * S_b[p, q] with both scales read from the
                // group's int8 stage, released here once they are read
                for (int k = 0; k < cu.nst / 2; ++k, ++g) {
                    const int buf = g % CF::kNbuf;
                    const int s8 = g % S8;
                    int ok = 0;
                    if (lane == 0) ok = bounded_wait(&tfull[buf], (g / CF::kNbuf) & 1, abort_flag, limit);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) continue;
                    tc::tc_fence_after_sync();
                    const uint32_t xs8 = sbase + CF::kOffXS + s8 * CF::kXS;
                    const uint32_t ys8 = sbase + CF::kOffYS + s8 * CF::kYS;
                    float4 xv;  // xs[p, b] for the group's four blocks
                    if (prm.xs_sb == 1) {
                        xv = tc::lds128f(xs8 + prow * (GROUP * 4));
                    } else {
                        xv.x = tc::lds32f(xs8 + (prow * prm.xs_sr + 0 * prm.xs_sb) * 4);
                        xv.y = tc::lds32f(xs8 + (prow * prm.xs_sr + 1 * prm.xs_sb) * 4);
                        xv.z = tc::lds32f(xs8 + (prow * prm.xs_sr + 2 * prm.xs_sb) * 4);
                        xv.w = tc::lds32f(xs8 + (prow * prm.xs_sr + 3 * prm.xs_sb) * 4);
                    }
                    const uint64_t x0 = f2_pack(__float_as_uint(xv.x), __float_as_uint(xv.x));
                    const uint64_t x1 = f2_pack(__float_as_uint(xv.y), __float_as_uint(xv.y));
                    const uint64_t x2 = f2_pack(__float_as_uint(xv.z), __float_as_uint(xv.z));
                    const uint64_t x3 = f2_pack(__float_as_uint(xv.w), __float_as_uint(xv.w));
                    const uint32_t ts = t_lane + static_cast<uint32_t>(buf * CF::kBufCols + cb);
#pragma unroll
                    for (int c = 0; c < NCH; ++c) {
                        uint32_t sv[GROUP][CF::kCH];
#pragma unroll
                        for (int b = 0; b < GROUP; ++b) tc::TmemLd<CF::kCH>::load(ts + b * BN + c * CF::kCH, sv[b]);
#pragma unroll
                        for (int b = 0; b < GROUP; ++b) tc::TmemLd<CF::kCH>::wait(sv[b]);
#pragma unroll
                        for (int t = 0; t < CF::kCH; t += 2) {
                            // ys[q, 0..3] of columns q, q + 1: one row of the [BN][4] scale tile each
                            const int q = cb + c * CF::kCH + t;
                            const float4 y0 = tc::lds128f(ys8 + q * (GROUP * 4));
                            const float4 y1 = tc::lds128f(ys8 + (q + 1) * (GROUP * 4));
                            const int a = (c * CF::kCH + t) / 2;
                            uint64_t r = acc[a];
                            r = f2_fma(f2_mul(x0, f2_pack(__float_as_uint(y0.x), __float_as_uint(y1.x))),
                                       f2_pack(sv[0][t], sv[0][t + 1]), r);
                            r = f2_fma(f2_mul(x1, f2_pack(__float_as_uint(y0.y), __float_as_uint(y1.y))),
                                       f2_pack(sv[1][t], sv[1][t + 1]), r);
                            r = f2_fma(f2_mul(x2, f2_pack(__float_as_uint(y0.z), __float_as_uint(y1.z))),
                                       f2_pack(sv[2][t], sv[2][t + 1]), r);
                            r = f2_fma(f2_mul(x3, f2_pack(__float_as_uint(y0.w), __float_as_uint(y1.w))),
                                       f2_pack(sv[3][t], sv[3][t + 1]), r);
                            acc[a] = r;
                        }
                    }
                    tc::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        tc::mbar_arrive(&tempty[buf]);
                        tc::mbar_arrive(&empty8[s8]);
                    }
                }
            } else {
                for (int k = 0; k < nblk; ++k, ++g) {
                    const int buf = g % CF::kNbuf;
                    int ok = 0;
                    if (lane == 0) ok = bounded_wait(&tfull[buf], (g / CF::kNbuf) & 1, abort_flag, limit);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) continue;
                    tc::tc_fence_after_sync();
                    const uint32_t ts = t_lane + static_cast<uint32_t>(buf * 2 * BN + cb);
                    if constexpr (SUMS) {
                        const int64_t b = static_cast<int64_t>(cu.g_begin) * GROUP + k;
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            uint32_t sv[CF::kCH];
                            tc::TmemLd<CF::kCH>::load(ts + c * CF::kCH, sv);
                            tc::TmemLd<CF::kCH>::wait(sv);
                            if (pv) {
#pragma unroll
                                for (int t = 0; t < CF::kCH; ++t) {
                                    const int64_t q = cu.q0 + cb + c * CF::kCH + t;
                                    if (q < prm.Q)
                                        prm.S[p * prm.sp + q * prm.sq + b] = static_cast<int32_t>(__uint_as_float(sv[t]));
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < NCH; ++c) {
                            uint32_t sv[CF::kCH], pvv[CF::kCH];
                            tc::TmemLd<CF::kCH>::load(ts + c * CF::kCH, sv);
                            tc::TmemLd<CF::kCH>::load(ts + BN + c * CF::kCH, pvv);
                            tc::TmemLd<CF::kCH>::wait(sv);
                            tc::TmemLd<CF::kCH>::wait(pvv);
#pragma unroll
                            for (int t = 0; t < CF::kCH; t += 2) {
                                const int a = (c * CF::kCH + t) / 2;
                                acc[a] = f2_fma(f2_pack(pvv[t], pvv[t + 1]), f2_pack(sv[t], sv[t + 1]), acc[a]);
                            }
                        }
                    }
                    tc::tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&tempty[buf]);
                }
            }
            // the tile's last unit on this CTA: write it and start the next from zero
            const bool tile_end = !ESC || u + 1 >= u_end || (u + 1) / prm.splits != u / prm.splits;
            if constexpr (!SUMS) {
                if (tile_end && *abort_flag == 0 && pv) {
                    float accf[CF::kCW];
#pragma unroll
                    for (int t = 0; t < CF::kCW / 2; ++t) {
                        accf[2 * t] = __uint_as_float(static_cast<uint32_t>(acc[t]));
                        accf[2 * t + 1] = __uint_as_float(static_cast<uint32_t>(acc[t] >> 32));
                    }
                    if (prm.vec_store) {
#pragma unroll
                        for (int t = 0; t < CF::kCW; t += 4) {
                            const int64_t q = cu.q0 + cb + t;
                            if (q < prm.Q)
                                *reinterpret_cast<float4*>(prm.C + p * prm.ldp + q) =
                                    make_float4(accf[t], accf[t + 1], accf[t + 2], accf[t + 3]);
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < CF::kCW; ++t) {
                            const int64_t q = cu.q0 + cb + t;
                            if (q < prm.Q) {
                                float* dst = prm.C + p * prm.ldp + q * prm.ldq;
                                if (prm.atomic)
                                    atomicAdd(dst, accf[t]);
                                else
                                    *dst = accf[t];
                            }
                        }
                    }
                }
                if (tile_end) {
#pragma unroll
                    for (int t = 0; t < CF::kCW / 2; ++t) acc[t] = 0ull;
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

// Zeroes C before a split-K contraction adds its partial tiles.  A kernel
// rather than a memset node, so that it takes part in the programmatic
// dependent launches: it starts while the previous kernel runs, and the
// contraction kernel's prologue overlaps it.
__global__ void __launch_bounds__(256) zero_f32_kernel(float* __restrict__ p, int64_t n) {
    pdl_wait();  // the previous kernel may still read or write C
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.0f;
}

// Pre-tiles the activation operand X = A [P, K] (with its scales AS [P, K/32])
// for the PREX kernels: one CTA per (128-row tile, 64-K f16 stage) writes the
// stage's f16 tile in the UMMA K-major 128-byte-swizzle layout (row r at r * 128
// bytes, its 16-byte chunk j at ((j ^ (r & 7)) << 4)) and the scale-product
// operands of the stage's two Q8_0 blocks (row r's 16 bf16 [h h h m m m l l l
// 0 ..] at (r >> 3) * 256 + (r & 7) * 16, the second K half 128 bytes on), i.e.
// exactly what the converter warps would write into the f16 ring.  Rows past P
// are zero.  Every 128-row tile is then converted once per call instead of once
// per output-column tile.
__global__ void __launch_bounds__(256)
tile_x_kernel(const int8_t* __restrict__ A, const float* __restrict__ AS, uint8_t* __restrict__ T, int64_t P,
              int64_t K) {
    pdl_trigger();
    pdl_wait();
    const int64_t ns = K / KS;
    const int64_t KB = K / 32;
    const int64_t tile = blockIdx.x / ns, st = blockIdx.x % ns;
    uint8_t* out = T + static_cast<int64_t>(blockIdx.x) * kXtStage;
    for (int i = threadIdx.x; i < BM * 8; i += blockDim.x) {
        const int r = i >> 3, j = i & 7;
        const int64_t p = tile * BM + r;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (p < P) {
            const uint2 b = *reinterpret_cast<const uint2*>(A + p * K + st * KS + j * 8);
            i8x4_to_f16x4(b.x, o.x, o.y);
            i8x4_to_f16x4(b.y, o.z, o.w);
        }
        *reinterpret_cast<uint4*>(out + r * (KS * 2) + ((j ^ (r & 7)) << 4)) = o;
    }
    for (int i = threadIdx.x; i < BM * 2; i += blockDim.x) {
        const int r = i % BM, bb = i / BM;
        const int64_t p = tile * BM + r;
        const float sc = p < P ? AS[p * KB + st * 2 + bb] : 0.0f;
        uint32_t sh, sm, sl3;
        split3_bf16(sc, sh, sm, sl3);
        uint8_t* dst = out + kXtF16 + bb * (BM * 32) + (r >> 3) * 256 + (r & 7) * 16;
        *reinterpret_cast<uint4*>(dst) = make_uint4(sh | (sh << 16), sh | (sm << 16), sm | (sm << 16), sl3 | (sl3 << 16));
        *reinterpret_cast<uint4*>(dst + 128) = make_uint4(sl3, 0u, 0u, 0u);
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

// int8 [rows, K] row-major, box {128 bytes of K, box_rows}, 128-byte swizzle,
// zero fill outside the tensor (ragged rows read as 0).  Boxes of 16 KB and
// more keep the TMA unit's few outstanding operations per SM busy enough to
// stream from HBM at full rate.
bool make_i8_map(CUtensorMap* map, const int8_t* base, int64_t rows, int64_t K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(KS8), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q5_0 weight rows [rows, K/32 * 20] bytes, box {80 bytes = one scale group,
// box_rows}, no swizzle, zero fill outside (ragged rows read as 0).
bool make_q5_map(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t row_bytes, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kQ5Row), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// f32 plane [outer, inner] with the given row stride in bytes, box {box_inner,
// box_outer}, no swizzle, zero fill outside.
bool make_f32_map(CUtensorMap* map, const float* base, int64_t inner, int64_t outer, int64_t stride_bytes,
                  int box_inner, int box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

constexpr int kMaxDevices = 64;

DeviceInfo device_info(int dev) {
    static std::mutex mu;
    static DeviceInfo cache[kMaxDevices];
    static bool have[kMaxDevices] = {};
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

template <int BN, int NCONV, int NEPI, int S8, int S16, int MINB, bool SUMS, bool PREX = false, bool Q5 = false,
          bool ESC = false>
cudaError_t launch_cfg(const CUtensorMap* maps, const TcParams& prm, int64_t grid, cudaStream_t stream) {
    using CF = Cfg<BN, NCONV, NEPI, S8, S16, Q5, ESC>;
    auto kern = qdot_tc_kernel<BN, NCONV, NEPI, S8, S16, MINB, SUMS, PREX, Q5, ESC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, CF::kSmem);
    if (e != cudaSuccess) return e;
    // the register split adds up only if every thread was launched with 128 registers
    static const int regs = [&] {
        cudaFuncAttributes fa{};
        return cudaFuncGetAttributes(&fa, kern) == cudaSuccess ? fa.numRegs : 0;
    }();
    TcParams p = prm;
    p.regsplit = (CF::kThreads == 512 && CF::kE0 == 8 && regs == 128) ? 1 : 0;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(CF::kThreads), static_cast<size_t>(CF::kSmem),
                      stream, maps[0], maps[1], maps[2], maps[3], p);
}

// Q5 = true: a.W holds Q5_0 weight blocks [N, K/32 * 20] bytes (q50_qdot_t);
// only the prompt layout (M > 64, X = A, Y = W) and not in block-sum mode.
template <bool SUMS, bool Q5 = false>
cudaError_t launch_tc(const QdotArgs& a, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorNotSupported;
    const DeviceInfo info = device_info(dev);
    if (!info.ok) return cudaErrorNotSupported;
    if (a.K % (KS * 2) != 0) return cudaErrorNotSupported;
    if (a.K > 0x7fffffffLL || a.M > 0x7fffffffLL || a.N > 0x7fffffffLL) return cudaErrorNotSupported;
    const int64_t KB = a.K / 32;
    const bool swap = a.M <= 64;
    if (Q5 && (SUMS || swap || (reinterpret_cast<uintptr_t>(a.W) & 15u) != 0)) return cudaErrorNotSupported;
    TcParams prm{};
    const int64_t P = swap ? a.N : a.M;
    const int64_t Q = swap ? a.M : a.N;
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
    // Persistent CTAs, one per SM, take the work units round-robin.  K is split
    // when the tiles are too few for the SMs: the smallest split count whose
    // units spread evenly (the busiest SM within ~5% of the mean), each split
    // keeping at least two scale groups.
    const int64_t tiles = gx * gy;
    const int64_t sms = info.sms;
    int splits = 1;
    if (tiles < 4 * sms) {
        for (int s = 1; s <= std::max(1, ngroups / 2); ++s) {
            const int64_t units = tiles * s;
            const double per_sm = static_cast<double>(units) / sms;
            const int64_t busiest = (units + sms - 1) / sms;
            splits = s;
            if (units >= sms && busiest <= per_sm * 1.05 + 1e-9) break;
        }
    }
    prm.groups_per_split = (ngroups + splits - 1) / splits;
    splits = (ngroups + prm.groups_per_split - 1) / prm.groups_per_split;
    if (tiles * splits > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    prm.splits = splits;
    prm.tiles_p = static_cast<int>(gx);
    prm.units = static_cast<int>(tiles * splits);
    const int64_t grid = std::min<int64_t>(prm.units, sms);
    prm.atomic = (!SUMS && splits > 1) ? 1 : 0;
    prm.vec_store = (!SUMS && !swap && !prm.atomic && (Q % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(a.C) & 15u) == 0) ? 1 : 0;

    CUtensorMap maps[4];
    const int8_t* X = swap ? a.W : a.A;
    const int8_t* Y = swap ? a.A : a.W;
    if (!make_i8_map(&maps[0], X, P, a.K, BM)) return cudaErrorInvalidValue;
    if (Q5 ? !make_q5_map(&maps[1], reinterpret_cast<const uint8_t*>(Y), Q, KB * kQ5Block, BN)
           : !make_i8_map(&maps[1], Y, Q, a.K, BN))
        return cudaErrorInvalidValue;
    prm.has_scales = SUMS ? 0 : 1;
    if (!SUMS) {
        // scale planes by TMA: rows of 16-byte multiples from a 16-byte aligned base
        auto plane = [&](CUtensorMap* m, const float* base, int64_t r_stride, int64_t b_stride, int64_t rows,
                         int box_rows, int& sr, int& sb) -> cudaError_t {
            if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0) return cudaErrorNotSupported;
            if (b_stride == 1) {  // [rows, KB]: box {4 blocks, box_rows} -> smem [row][4]
                if ((r_stride * 4) % 16 != 0) return cudaErrorNotSupported;
                sr = GROUP; sb = 1;
                return make_f32_map(m, base, KB, rows, r_stride * 4, GROUP, box_rows) ? cudaSuccess
                                                                                     : cudaErrorInvalidValue;
            }
            // [KB, rows]: box {box_rows, 4 blocks} -> smem [4][row]
            if ((b_stride * 4) % 16 != 0) return cudaErrorNotSupported;
            sr = 1; sb = box_rows;
            return make_f32_map(m, base, rows, KB, b_stride * 4, box_rows, GROUP) ? cudaSuccess
                                                                                 : cudaErrorInvalidValue;
        };
        cudaError_t e1 = plane(&maps[2], prm.xs, prm.xs_r, prm.xs_b, P, BM, prm.xs_sr, prm.xs_sb);
        if (e1 != cudaSuccess) return e1;
        e1 = plane(&maps[3], prm.ys, prm.ys_r, prm.ys_b, Q, BN, prm.ys_sr, prm.ys_sb);
        if (e1 != cudaSuccess) return e1;
    } else {
        maps[2] = maps[0];
        maps[3] = maps[1];
    }
    // Pre-tiled X for the prompt shapes (X = A): converted once per call into a
    // per-(device, stream) workspace, unless the caller allocates nothing or the
    // workspace cannot be had now (stream capture); then the converter warps
    // convert X in the kernel as for every other shape.
    bool prex = false;
    if (!SUMS && !swap && a.no_alloc == 0) {
        const int64_t ns = a.K / KS;
        const int64_t tp = (P + BM - 1) / BM;
        void* xt = nullptr;
        if (tp * ns <= 0x7fffffffLL &&
            stream_workspace(stream, static_cast<size_t>(tp * ns) * kXtStage, &xt) == cudaSuccess) {
            cudaError_t e0 = launch_pdl(tile_x_kernel, dim3(static_cast<unsigned>(tp * ns)), dim3(256), 0, stream,
                                        a.A, a.AS, static_cast<uint8_t*>(xt), P, a.K);
            if (e0 != cudaSuccess) return e0;
            prm.xt = static_cast<const uint8_t*>(xt);
            prm.xt_tile_stride = ns * kXtStage;
            prex = true;
        }
    }
    cudaError_t e = cudaSuccess;
    if (prm.atomic) {
        const int64_t n = a.M * a.N;
        const int64_t blocks = std::min<int64_t>((n + 1023) / 1024, 2 * sms);
        e = launch_pdl(zero_f32_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a.C, n);
        if (e != cudaSuccess) return e;
    }
    // six converter warps (measured 8 % faster than four at M = 512; eight
    // spill) and ring depths (int8 stages S8, f16 stages S16) within 227 KB of
    // shared memory: three f16 stages measured ~11 % faster than two at every
    // shape (the converters run ahead of the MMA issuer), at the cost of int8
    // depth
    if constexpr (Q5) {
        if (prex) return launch_cfg<128, 6, 8, 2, 3, 1, false, true, true>(maps, prm, grid, stream);
        return launch_cfg<128, 6, 8, 2, 3, 1, false, false, true>(maps, prm, grid, stream);
    }
    if (!swap) {
        if constexpr (!SUMS)
            if (prex) return launch_cfg<128, 6, 8, 2, 3, 1, SUMS, true>(maps, prm, grid, stream);
        return launch_cfg<128, 6, 8, 2, 3, 1, SUMS>(maps, prm, grid, stream);
    }
    if constexpr (SUMS) {
        if (BN == 16) return launch_cfg<16, 6, 8, 5, 3, 1, SUMS>(maps, prm, grid, stream);
        if (BN == 32) return launch_cfg<32, 6, 8, 5, 3, 1, SUMS>(maps, prm, grid, stream);
        return launch_cfg<64, 6, 8, 4, 3, 1, SUMS>(maps, prm, grid, stream);
    } else {
        // narrow tiles take the scales in the epilogue (the activation scale tile is
        // [BN][4] in shared memory here: AS is row-major); the int8 ring is then
        // deeper, as each stage lives until the epilogue has read its scales
        if (prm.ys_sr != GROUP || prm.ys_sb != 1) return cudaErrorNotSupported;
        if (BN == 16) return launch_cfg<16, 6, 8, 8, 3, 1, false, false, false, true>(maps, prm, grid, stream);
        if (BN == 32) return launch_cfg<32, 6, 8, 7, 3, 1, false, false, false, true>(maps, prm, grid, stream);
        return launch_cfg<64, 6, 8, 5, 3, 1, false, false, false, true>(maps, prm, grid, stream);
    }
}

}  // namespace

int g_prompt_kernel = 1;  // 1: the kernel of qdot_tcw.cu where it applies; 0: this file's kernel

void set_prompt_kernel(int which) { g_prompt_kernel = which; }

cudaError_t launch_qdot_tc(const QdotArgs& a, cudaStream_t stream) {
    if (a.S == nullptr && a.M > 64 && g_prompt_kernel == 1) {
        const cudaError_t e = launch_qdot_tcw(a, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    return a.S != nullptr ? launch_tc<true>(a, stream) : launch_tc<false>(a, stream);
}

cudaError_t launch_qdot_tc_q50(const QdotArgs& a, cudaStream_t stream) {
    if (a.S != nullptr) return cudaErrorNotSupported;
    if (a.M > 64 && g_prompt_kernel == 1) {
        const cudaError_t e = launch_qdot_tcw(a, stream, true);
        if (e != cudaErrorNotSupported) return e;
    }
    return launch_tc<false, true>(a, stream);
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
