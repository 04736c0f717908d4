// qdot_t for prompt-sized M on the sm_103a tensor cores, with the scales
// applied in f32 registers (no scale-product MMA) and two Q8_0 blocks per
// hand-off between the roles; also q50_qdot_t, with Q5_0 weight blocks.
//
// What it computes ("Quantized built-ins and formats", section "Q8_0"; the
// integer-tensor-core variant qmma_t in "Phobos Language Spec" section 10):
//   out[i, j] = sum_b a_scales[i, b] * w_scales[j, b] * S[i, j, b],
//   S[i, j, b] = sum_{k in block b} a[i, k] * w[j, k]   (an integer),
// with w[j, k] = q - 16 for Q5_0 weights ("Phobos Language Spec" section 10,
// Q5_0 row).
//
// Engine.  As in the other tensor-core kernel: int8 values are exact in f16,
// and every partial sum of one 32-element block (|S| <= 2^19 < 2^24) is exact
// in the f32 accumulator, so two K = 16 kind::f16 MMAs into a fresh TMEM
// buffer give the block sums S exactly.  The epilogue warps apply the scales
// in f32 registers: acc[j, i] += w_scale[j] * (a_scale[i] * S).
//
// Orientation.  The MMA's 128-row side (TMEM lanes) is a tile of 128 weight
// rows j; its N = 128 side is a tile of 128 activation rows i.  So a weight
// scale is one value per TMEM lane (per epilogue thread row) and an
// activation scale one value per column, and the activation scales can be laid
// out in the order the epilogue threads read them.  The weights are widened
// int8 -> f16 (or Q5_0 blocks decoded to q - 16 in f16) by four converter warps
// from the TMA-loaded tile into the f16 stage; the activations were converted
// once per call into f16 MMA tiles by a small kernel (tile_act_kernel) and
// arrive by bulk copy.
//
// Hand-offs.  One f16 stage holds 64 K (two Q8_0 blocks) of both operands,
// and one accumulator buffer of 256 TMEM columns holds the block sums of those
// two blocks (two buffers fill the 512 columns): the MMA issuer waits twice and
// commits twice per two blocks.  (A version with one block per hand-off and the
// weights in tensor memory was bound by the latency of its per-block hand-offs.)
//
// Warps (704 threads, one persistent CTA per SM over (activation tile, weight
// tile, K split) units, the activation tile fastest, so the CTAs running at
// the same time share weight tiles in L2):
//   warp 0      producer: per scale group (128 K) the weight tile and
//               the weight-scale box (TMA), the group's activation scales,
//               and the activation tiles of two f16 stages (bulk copies);
//   warp 1      MMA issuer (one thread), TMEM allocation;
//   warps 2..5  converters, 32 weight rows each;
//   warps 6..21 epilogue: four TMEM lane quadrants x four column quarters,
//               each thread holding 4 weight rows x 8 activation rows of the
//               accumulator tile in registers; the unit's end stores C.
//
// Safety.  Every mbarrier wait is bounded (a clock64 limit).  A wait that
// gives up sets this file's device status word and a CTA-wide abort flag;
// every role then runs out its loops without waiting or working, copies and
// MMAs in flight are drained with bounded waits, TMEM is freed and the kernel
// returns.  The host reads the status through read_and_clear_status_w.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "pq.h"
#include "pq_device.cuh"
#include "pq_internal.h"
#include "tc_ptx.cuh"

namespace pq {

// Nonzero after a bounded on-device wait of this kernel gave up.
__device__ unsigned g_pq_status_w;

namespace {

constexpr int TW = 128;                  // weight rows per tile (MMA M, TMEM lanes)
constexpr int TA = 128;                  // activation rows per tile (MMA N)
constexpr int GROUP = 4;                 // Q8_0 blocks per scale group (128 K)
constexpr int kNbufD = 2;                // accumulator buffers of two blocks each (256 columns)
constexpr int kAct = TA * 64 * 2;        // f16 activation tile of one stage: 128 rows x 64 K (16 KB)
constexpr int kWt = TW * 64 * 2;         // f16 weight tile of one stage: 128 rows x 64 K (16 KB)
constexpr int kStage = kAct + kWt;       // one f16 stage: two Q8_0 blocks of both operands
constexpr int kAsc = GROUP * TA * 4;     // activation scales of one group (2 KB)
constexpr int kW8 = TW * 128;            // weight tile slot of one group: int8 (16 KB) or Q5_0 (10 KB)
constexpr int kQ5Row = GROUP * 20;       // Q5_0 blocks of one row and group: 4 x (qh word + 16 nibble bytes)
constexpr int kWsc = TW * GROUP * 4;     // weight scales of one group (2 KB)
constexpr int S16 = 4;                   // f16 stages
constexpr int S8 = 3;                    // weight tile stages (groups)
constexpr int SR = 4;                    // scale slots (groups)
constexpr int kOffSt = 0;
constexpr int kOffW8 = kOffSt + S16 * kStage;
constexpr int kOffSc = kOffW8 + S8 * kW8;          // slot: weight scales, then activation scales
constexpr int kSc = kWsc + kAsc;
constexpr int kOffBar = kOffSc + SR * kSc;
constexpr int kNumBars = 2 * S16 + 2 * S8 + 2 * SR + 2 * kNbufD + 1;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmem = kOffMisc + 16 + 1024;        // + alignment slack
constexpr int kThreads = 704;            // 22 warps
constexpr int kConv0 = 2;                // first converter warp
constexpr int kEpi0 = 6;                 // first epilogue warp (16 of them)
constexpr int kNepi = 16;
constexpr unsigned kBackoff = 64;        // ns between failed barrier tests of the waiting roles
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kAct % 1024 == 0 && kWt % 1024 == 0 && kW8 % 1024 == 0 && kSc % 1024 == 0, "1024-byte aligned tiles");

struct TcwParams {
    float* C;                  // C[i * N + j], [M, N] row-major
    int64_t M, N, K;
    int ngroups;               // K / 128
    int groups_per_split;
    int splits;                // K splits per tile
    int tiles_a;               // activation tiles
    int units;                 // tiles_a * tiles_w * splits
    int atomic;                // split-K: red.add into a zeroed C
    int ws_rowmajor;           // 1: WS [N, K/32] (smem [row][4]); 0: WS [K/32, N] (smem [4][row])
    const uint8_t* act;        // f16 activation stages: [tiles_a][K / 64] x kAct bytes
    const uint8_t* asc;        // activation scales: [tiles_a][ngroups] x kAsc bytes
    int inject_skip_stage;     // test hook: the producer skips this group (-1: off)
    unsigned long long timeout_cycles;
};

__device__ __forceinline__ void set_abort(volatile int* abort_flag) {
    if (*abort_flag == 0) {
        *abort_flag = 1;
        atomicOr(&g_pq_status_w, 1u);
    }
}

// Waits for the phase of `bar` with the given parity; false if the CTA is
// aborting or the wait ran past its limit (which starts the abort).  After a
// failed test the thread sleeps about `backoff_ns` before the next, so that a
// role that is waiting leaves the issue slots of its SM sub-partition to the
// epilogue warps, which bound the kernel (0: test again at once).
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned long long limit, unsigned backoff_ns = 0) {
    if (*abort_flag) return false;
    if (tc::mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (backoff_ns) __nanosleep(backoff_ns);
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
            atomicOr(&g_pq_status_w, 2u);
            return;
        }
    }
}

// Warp-uniform bounded wait: lane 0 waits, the result is broadcast.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long limit, int lane, unsigned backoff_ns = 0) {
    int ok = 0;
    if (lane == 0) ok = bounded_wait(bar, parity, abort_flag, limit, backoff_ns);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Waits for every tcgen05.ld this thread has issued; the 8 registers named are
// those of the load it is meant for, so no use of them is scheduled before it.
__device__ __forceinline__ void tmem_wait_ld8(uint32_t (&r)[8]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7])
                 :
                 : "memory");
}

// Q5_0 ("Phobos Language Spec" section 10, Q5_0 row): a block is the qh word,
// then 16 bytes whose byte e holds element e in its low nibble and element
// e + 16 in its high nibble, each element q - 16 with the fifth bit of q in
// bit e of qh.  q5_spread4 puts the four bits of x at bit 0 of the four bytes
// (x * 0x00204081 places bit i at bit 8i, no carries); q5_to_f16x4 turns four
// biased elements q in [0, 31] (one a byte) into two f16x2 of q - 16, exactly
// (each byte placed under the f16 exponent of 1024, then 1040 = 1024 + 16
// subtracted).
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

// The 16-byte f16 chunk c (elements 8c .. 8c + 7) of a Q5_0 block given as
// its qh word and four data words.
__device__ __forceinline__ uint4 q5_chunk(uint32_t qh, const uint32_t (&d)[4], int c) {
    uint32_t u[2];
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
        const int e0 = 8 * c + 4 * hw;  // first element of the word
        const uint32_t dw = d[(e0 & 15) >> 2];
        const uint32_t nib = e0 < 16 ? (dw & 0x0f0f0f0fu) : ((dw >> 4) & 0x0f0f0f0fu);
        u[hw] = nib | (q5_spread4((qh >> e0) & 0xfu) << 4);
    }
    uint4 o;
    q5_to_f16x4(u[0], o.x, o.y);
    q5_to_f16x4(u[1], o.z, o.w);
    return o;
}

// The epilogue's wait: every lane tests the barrier (no branch to lane 0 and no
// broadcast); the result is made warp-uniform before the warp-collective TMEM
// loads it guards.  The abort flag is read from shared memory by its address.
__device__ __forceinline__ uint32_t abort_get(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ bool epi_wait(uint64_t* bar, uint32_t parity, uint32_t abort_a, unsigned long long limit) {
    bool ok = abort_get(abort_a) == 0;
    if (ok && !tc::mbar_try_wait(bar, parity)) {
        const long long t0 = clock64();
        for (uint32_t n = 1;; ++n) {
            if (tc::mbar_try_wait(bar, parity)) break;
            if ((n & 31) == 0) {
                if (abort_get(abort_a)) {
                    ok = false;
                    break;
                }
                if (static_cast<unsigned long long>(clock64() - t0) > limit) {
                    set_abort(reinterpret_cast<volatile int*>(__cvta_shared_to_generic(abort_a)));
                    ok = false;
                    break;
                }
            }
        }
    }
    return __all_sync(0xffffffffu, ok);
}

// Arrival on a barrier by lane 0 of the warp, as one predicated instruction.
__device__ __forceinline__ void arrive_lane0(uint64_t* bar, int lane) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.eq.s32 p, %1, 0;\n\t"
                 "@p mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];\n\t}"
                 ::"r"(tc::smem_u32(bar)), "r"(lane) : "memory");
}

// NREG registers a thread (the launcher takes the largest build the device
// admits with 704 threads); WSR: weight scales [N, K/32] (else [K/32, N]); Q5:
// the weights are Q5_0 blocks [N, K/32 * 20] bytes (q50_qdot_t) instead of int8
template <int NREG, bool WSR, bool Q5>
__global__ void __maxnreg__(NREG)
qdot_tcw_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWS,
                const TcwParams prm) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint64_t* full16 = bars;                  // f16 stage ready: activations landed (tx) + 4 converter warps
    uint64_t* empty16 = full16 + S16;         // its MMAs completed (commit)
    uint64_t* full8 = empty16 + S16;          // weight tile landed (producer, tx)
    uint64_t* empty8 = full8 + S8;            // converted (4 converter warps)
    uint64_t* sfull = empty8 + S8;            // scales of a group landed (producer, tx)
    uint64_t* sempty = sfull + SR;            // read (16 epilogue warps)
    uint64_t* tfull = sempty + SR;            // block sums of a pair of blocks in an accumulator buffer (commit)
    uint64_t* tempty = tfull + kNbufD;        // read (16 epilogue warps)
    uint64_t* drain = tempty + kNbufD;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    const uint32_t sbase = tc::smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long limit = prm.timeout_cycles;

    // work unit u -> (activation tile, weight tile, K split) and its scale groups
    struct Unit {
        int a_tile;
        int64_t i0, j0;   // first activation row, first weight row
        int g_begin, ng;
    };
    auto unit = [&](int u) {
        Unit r;
        const int z = u % prm.splits;
        const int t = u / prm.splits;
        r.a_tile = t % prm.tiles_a;
        r.i0 = static_cast<int64_t>(r.a_tile) * TA;
        r.j0 = static_cast<int64_t>(t / prm.tiles_a) * TW;
        r.g_begin = z * prm.groups_per_split;
        r.ng = max(0, min(prm.ngroups, r.g_begin + prm.groups_per_split) - r.g_begin);
        return r;
    };
    const int u_first = static_cast<int>(blockIdx.x);
    const int u_step = static_cast<int>(gridDim.x);

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int i = 0; i < S16; ++i) {
            tc::mbar_init(&full16[i], 1 + 4);
            tc::mbar_init(&empty16[i], 1);
        }
        for (int i = 0; i < S8; ++i) {
            tc::mbar_init(&full8[i], 1);
            tc::mbar_init(&empty8[i], 4);
        }
        for (int i = 0; i < SR; ++i) {
            tc::mbar_init(&sfull[i], 1);
            tc::mbar_init(&sempty[i], kNepi);
        }
        for (int i = 0; i < kNbufD; ++i) {
            tc::mbar_init(&tfull[i], 1);
            tc::mbar_init(&tempty[i], kNepi);
        }
        tc::mbar_init(drain, 1);
        *abort_flag = 0;
        tc::fence_mbar_init();
        tc::tma_prefetch_map(&tmW);
        tc::tma_prefetch_map(&tmWS);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
        tc::tc_fence_before_sync();
    }
    __syncthreads();
    tc::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // everything below reads global memory the preceding kernel may have written
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int gi = 0;  // scale groups over all units of this CTA
            int issued8 = 0, issuedS = 0, issued16 = 0;
            for (int u = u_first; u < prm.units; u += u_step) {
                const Unit un = unit(u);
                for (int k = 0; k < un.ng; ++k, ++gi) {
                    const int g = un.g_begin + k;
                    if (gi == prm.inject_skip_stage) continue;  // test hook: this group never arrives
                    // weight tile of the group: 128 rows x 128 K, int8 with 128-byte swizzle
                    // or Q5_0 blocks (80 bytes a row, no swizzle)
                    const int s8 = gi % S8;
                    if (bounded_wait(&empty8[s8], ((gi / S8) & 1) ^ 1, abort_flag, limit, kBackoff)) {
                        issued8 = gi + 1;
                        tc::mbar_arrive_expect_tx(&full8[s8], Q5 ? TW * kQ5Row : kW8);
                        tc::tma_load_2d(smem + kOffW8 + s8 * kW8, &tmW, &full8[s8], g * (Q5 ? kQ5Row : 128),
                                        static_cast<int>(un.j0));
                    }
                    // weight scales (TMA box) and activation scales (bulk copy) of the group
                    const int sr = gi % SR;
                    if (bounded_wait(&sempty[sr], ((gi / SR) & 1) ^ 1, abort_flag, limit, kBackoff)) {
                        issuedS = gi + 1;
                        tc::mbar_arrive_expect_tx(&sfull[sr], kSc);
                        const int b0 = g * GROUP;
                        tc::tma_load_2d(smem + kOffSc + sr * kSc, &tmWS, &sfull[sr],
                                        prm.ws_rowmajor ? b0 : static_cast<int>(un.j0),
                                        prm.ws_rowmajor ? static_cast<int>(un.j0) : b0);
                        tc::bulk_copy_g2s(smem + kOffSc + sr * kSc + kWsc,
                                          prm.asc + (static_cast<int64_t>(un.a_tile) * prm.ngroups + g) * kAsc, kAsc,
                                          &sfull[sr]);
                    }
                    // the activation tiles of the group's two f16 stages
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const int si = 2 * gi + h;
                        const int s16 = si % S16;
                        if (!bounded_wait(&empty16[s16], ((si / S16) & 1) ^ 1, abort_flag, limit, kBackoff)) continue;
                        issued16 = si + 1;
                        tc::mbar_arrive_expect_tx(&full16[s16], kAct);
                        tc::bulk_copy_g2s(smem + kOffSt + s16 * kStage,
                                          prm.act + (static_cast<int64_t>(un.a_tile) * (2 * prm.ngroups) + 2 * g + h) *
                                                        kAct,
                                          kAct, &full16[s16]);
                    }
                }
            }
            // copies in flight land before the CTA may exit (the skipped test group excepted;
            // an f16 stage also waits for the converters, whose arrivals are not awaited here,
            // so the drain of the f16 ring waits for the bytes alone: a bounded wait that may
            // report a timeout only after an abort)
            for (int i = max(0, issued8 - S8); i < issued8; ++i)
                if (i != prm.inject_skip_stage) drain_wait(&full8[i % S8], (i / S8) & 1, limit);
            for (int i = max(0, issuedS - SR); i < issuedS; ++i)
                if (i != prm.inject_skip_stage) drain_wait(&sfull[i % SR], (i / SR) & 1, limit);
            for (int i = max(0, issued16 - S16); i < issued16; ++i)
                if (i / 2 != prm.inject_skip_stage) drain_wait(&full16[i % S16], (i / S16) & 1, limit);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // one f16 stage = two Q8_0 blocks = one hand-off: four K = 16 MMAs into the
        // two 128-column halves of one accumulator buffer, one commit for the epilogue
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(TW, TA);
            int si = 0;  // f16 stages over all units of this CTA
            for (int u = u_first; u < prm.units; u += u_step) {
                const int nst = unit(u).ng * 2;
                for (int k = 0; k < nst; ++k, ++si) {
                    const int s16 = si % S16;
                    const int buf = si % kNbufD;
                    bool ok = bounded_wait(&full16[s16], (si / S16) & 1, abort_flag, limit, kBackoff);
                    ok = ok && bounded_wait(&tempty[buf], ((si / kNbufD) & 1) ^ 1, abort_flag, limit, kBackoff);
                    if (ok) {
                        tc::tc_fence_after_sync();
                        const uint32_t a0 = sbase + kOffSt + s16 * kStage;  // activations: the MMA's B
                        const uint32_t w0 = a0 + kAct;                      // weights: the MMA's A
#pragma unroll
                        for (int bb = 0; bb < 2; ++bb)
#pragma unroll
                            for (int kk = 0; kk < 2; ++kk) {
                                const uint32_t koff = static_cast<uint32_t>((bb * 2 + kk) * 32);  // 16 f16 = 32 B
                                tc::umma_f16(tmem_base + static_cast<uint32_t>(buf * 2 * TA + bb * TA),
                                             tc::sw128_kmajor_desc(w0 + koff), tc::sw128_kmajor_desc(a0 + koff),
                                             idesc, kk);
                            }
                    }
                    // the commits arrive also after an abort, so that every barrier
                    // keeps a consistent phase for the drains
                    tc::umma_commit(&tfull[buf]);
                    tc::umma_commit(&empty16[s16]);
                }
            }
            tc::umma_commit(drain);  // arrives when every MMA issued above has completed
            drain_wait(drain, 0, limit);
        }
    } else if (warp >= kConv0 && warp < kEpi0) {
        // ------------------------------------------------------------ converters
        // warp cw widens weight rows 32 cw .. 32 cw + 31 of the group's weight tile, one row
        // per lane, into the f16 weight tiles of the group's two stages (UMMA K-major
        // 128-byte swizzle: row r at r * 128 bytes, 16-byte chunk c at (c ^ (r & 7)) << 4)
        const int row = (warp - kConv0) * 32 + lane;
        int gi = 0;
        for (int u = u_first; u < prm.units; u += u_step) {
            const int ng = unit(u).ng;
            for (int k = 0; k < ng; ++k, ++gi) {
                const int s8 = gi % S8;
                const bool ok8 = warp_wait(&full8[s8], (gi / S8) & 1, abort_flag, limit, lane, kBackoff);
                if constexpr (Q5) {
                    // the row's four Q5_0 blocks: 80 bytes (rows 80 bytes apart: the 16-byte
                    // loads of eight consecutive rows fall in distinct banks)
                    const uint32_t w5 = sbase + kOffW8 + s8 * kW8 + row * kQ5Row;
                    uint32_t q[GROUP * 5];
#pragma unroll
                    for (int t = 0; t < 5; ++t) {
                        const uint4 v = ok8 ? tc::lds128(w5 + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
                        q[4 * t] = v.x;
                        q[4 * t + 1] = v.y;
                        q[4 * t + 2] = v.z;
                        q[4 * t + 3] = v.w;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int si = 2 * gi + h;
                        const int s16 = si % S16;
                        const bool ok = ok8 && warp_wait(&empty16[s16], ((si / S16) & 1) ^ 1, abort_flag, limit,
                                                         lane, kBackoff);
                        if (ok) {
                            const uint32_t w16 = sbase + kOffSt + s16 * kStage + kAct + row * 128;
#pragma unroll
                            for (int bb = 0; bb < 2; ++bb) {
                                const int b = 2 * h + bb;  // block within the group
                                const uint32_t d[4] = {q[5 * b + 1], q[5 * b + 2], q[5 * b + 3], q[5 * b + 4]};
#pragma unroll
                                for (int c = 0; c < 4; ++c)
                                    tc::sts128(w16 + (((4 * bb + c) ^ (row & 7)) << 4), q5_chunk(q[5 * b], d, c));
                            }
                            tc::fence_proxy_async_smem();
                        }
                        __syncwarp();
                        // arrive also after an abort: every barrier keeps a consistent phase
                        if (lane == 0) tc::mbar_arrive(&full16[s16]);
                    }
                } else {
                    const uint32_t w8 = sbase + kOffW8 + s8 * kW8 + row * 128;
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const int si = 2 * gi + h;
                        const int s16 = si % S16;
                        const bool ok = ok8 && warp_wait(&empty16[s16], ((si / S16) & 1) ^ 1, abort_flag, limit,
                                                         lane, kBackoff);
                        if (ok) {
                            const uint32_t w16 = sbase + kOffSt + s16 * kStage + kAct + row * 128;
                            uint4 v[4];
#pragma unroll
                            for (int c = 0; c < 4; ++c) v[c] = tc::lds128(w8 + (((h * 4 + c) ^ (row & 7)) << 4));
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                uint4 o0, o1;
                                i8x4_to_f16x4(v[c].x, o0.x, o0.y);
                                i8x4_to_f16x4(v[c].y, o0.z, o0.w);
                                i8x4_to_f16x4(v[c].z, o1.x, o1.y);
                                i8x4_to_f16x4(v[c].w, o1.z, o1.w);
                                tc::sts128(w16 + (((2 * c) ^ (row & 7)) << 4), o0);
                                tc::sts128(w16 + (((2 * c + 1) ^ (row & 7)) << 4), o1);
                            }
                            tc::fence_proxy_async_smem();
                        }
                        __syncwarp();
                        // arrive also after an abort: every barrier keeps a consistent phase
                        if (lane == 0) tc::mbar_arrive(&full16[s16]);
                    }
                }
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&empty8[s8]);
            }
        }
    } else if (warp >= kEpi0) {
        // ------------------------------------------------------------ epilogue
        // thread (quadrant qd, column quarter cq, lane t): weight rows
        // 32 qd + t/4 + {0, 8, 16, 24} and activation rows 32 cq + 8 r + 2 (t % 4) + {0, 1},
        // r = 0..3, of the tile -- the 16x256b TMEM load layout over two 16-lane halves.
        // Every shared-memory and TMEM address below is a per-thread base plus a block
        // offset and a constant; the waits are taken by all lanes together and the
        // arrivals predicated on lane 0, without branches.
        const int qd = warp & 3;
        const int cq = (warp - kEpi0) >> 2;
        const int m = lane & 3;
        const int rr = lane >> 2;
        const uint32_t t_q = tmem_base + (static_cast<uint32_t>(qd * 32) << 16) + static_cast<uint32_t>(cq * 32);
        // weight scale of row 32 qd + rr + 8 k, block bb of a scale slot: [row][4] or [4][row]
        const uint32_t w_base = static_cast<uint32_t>(WSR ? (qd * 32 + rr) * GROUP * 4 : (qd * 32 + rr) * 4);
        constexpr uint32_t kWk = WSR ? 8 * GROUP * 4 : 8 * 4;
        constexpr uint32_t kWb = WSR ? 4 : TW * 4;
        // activation scales ordered [bb][cq][c][m][4]: one 16-byte load per chunk, the four
        // threads m of a chunk reading 64 contiguous bytes
        const uint32_t a_base = static_cast<uint32_t>(kWsc + (cq * 32 + m * 4) * 4);
        const uint32_t abort_a = tc::smem_u32(const_cast<int*>(abort_flag));
        uint64_t acc[4][4];  // [row k][r]: f32 pair of activation rows (2m, 2m + 1) + 8r + 32cq
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[k][r] = 0ull;
        uint32_t gi = 0;  // scale groups over all units of this CTA; stage 2 gi + h uses buffer h
        for (int u = u_first; u < prm.units; u += u_step) {
            const int ng = unit(u).ng;
            for (int kg = 0; kg < ng; ++kg, ++gi) {
                const uint32_t sr = gi % SR;
                const bool oks = epi_wait(&sfull[sr], (gi / SR) & 1, abort_a, limit);
                const uint32_t wsc = sbase + kOffSc + sr * kSc + w_base;
                const uint32_t asc = sbase + kOffSc + sr * kSc + a_base;
#pragma unroll 1
                for (int h = 0; h < kNbufD; ++h) {
                    const bool ok = oks && epi_wait(&tfull[h], gi & 1, abort_a, limit);
                    if (ok) {
                        tc::tc_fence_after_sync();
#pragma unroll 1
                        for (int bl = 0; bl < 2; ++bl) {
                            const int bb = h * 2 + bl;  // block within the group
                            uint64_t w2[4];             // weight scales of the thread's rows, as f32 pairs
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint32_t w = tc::lds32(wsc + k * kWk + bb * kWb);
                                w2[k] = f2_pack(w, w);
                            }
                            const uint32_t col0 = t_q + static_cast<uint32_t>(h * 2 * TA + bl * TA);
                            // sub-chunk s = 2 c + half: 16 columns of one 16-lane half; the load
                            // of sub-chunk s + 1 is issued before the arithmetic of sub-chunk s
                            float4 av = tc::lds128f(asc + bb * 512);
                            auto apply = [&](int sc, const uint32_t(&hv)[8]) {
                                const int c = sc >> 1, half = sc & 1;
#pragma unroll
                                for (int rl = 0; rl < 2; ++rl) {
                                    const int r = 2 * c + rl;
                                    const uint64_t a2 = rl ? f2_pack(__float_as_uint(av.z), __float_as_uint(av.w))
                                                           : f2_pack(__float_as_uint(av.x), __float_as_uint(av.y));
#pragma unroll
                                    for (int kk = 0; kk < 2; ++kk) {
                                        const int k = 2 * half + kk;
                                        acc[k][r] = f2_fma(w2[k], f2_mul(a2, f2_pack(hv[4 * rl + 2 * kk], hv[4 * rl + 2 * kk + 1])),
                                                           acc[k][r]);
                                    }
                                }
                            };
                            uint32_t hA[8], hB[8];
                            tc::TmemLd16x256bX2::load(col0, hA);
                            tmem_wait_ld8(hA);
                            tc::TmemLd16x256bX2::load(col0 + (16u << 16), hB);
                            apply(0, hA);
                            tmem_wait_ld8(hB);
                            tc::TmemLd16x256bX2::load(col0 + 16, hA);
                            apply(1, hB);
                            tmem_wait_ld8(hA);
                            av = tc::lds128f(asc + bb * 512 + 64);
                            tc::TmemLd16x256bX2::load(col0 + (16u << 16) + 16, hB);
                            apply(2, hA);
                            tmem_wait_ld8(hB);
                            if (bl == 1) {
                                // every load of this buffer has landed: hand it back
                                tc::tc_fence_before_sync();
                                __syncwarp();
                                arrive_lane0(&tempty[h], lane);
                            }
                            apply(3, hB);
                        }
                    } else {
                        tc::tc_fence_before_sync();
                        __syncwarp();
                        arrive_lane0(&tempty[h], lane);
                    }
                }
                __syncwarp();
                arrive_lane0(&sempty[sr], lane);
            }
            // the unit's tile (or K split of it) goes to C
            if (abort_get(abort_a) == 0) {
                const Unit un = unit(u);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int64_t j = un.j0 + qd * 32 + rr + 8 * k;
                    if (j < prm.N) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
#pragma unroll
                            for (int c = 0; c < 2; ++c) {
                                const int64_t i = un.i0 + cq * 32 + 8 * r + 2 * m + c;
                                const float v = __uint_as_float(c ? static_cast<uint32_t>(acc[k][r] >> 32)
                                                                  : static_cast<uint32_t>(acc[k][r]));
                                if (i < prm.M) {
                                    float* dst = prm.C + i * prm.N + j;
                                    if (prm.atomic)
                                        atomicAdd(dst, v);
                                    else
                                        *dst = v;
                                }
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[k][r] = 0ull;
        }
    }

    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after_sync();
        tc::tmem_dealloc(tmem_base, 512);
    }
}

// Converts the activations A [M, K] (with AS [M, K/32]) once per call into the
// layouts the kernel above copies into shared memory.  One CTA per (128-row
// activation tile, scale group of 128 K):
//   * two f16 stages of 64 K: row r of the tile at r * 128 bytes, its 16-byte
//     chunk c (K elements 8c .. 8c + 7) at ((c ^ (r & 7)) << 4) -- the UMMA
//     K-major 128-byte-swizzle layout of the MMA's B operand;
//   * the group's activation scales ordered [block b][column quarter cq][chunk q]
//     [m][e] for activation row 32 cq + 8 (2 q + e / 2) + 2 m + e % 2: an
//     epilogue thread (m = lane % 4) reads the four rows of its chunk q with one
//     16-byte load, the four threads m together 64 contiguous bytes.
// Rows past M are zero (their results are never stored).
__global__ void __launch_bounds__(256)
tile_act_kernel(const int8_t* __restrict__ A, const float* __restrict__ AS, uint8_t* __restrict__ act,
                float* __restrict__ asc, int64_t M, int64_t K) {
    pdl_trigger();
    pdl_wait();
    const int64_t ngroups = K / 128;
    const int64_t KB = K / 32;
    const int64_t tile = blockIdx.x / ngroups, g = blockIdx.x % ngroups;
    uint8_t* out = act + static_cast<int64_t>(blockIdx.x) * 2 * kAct;
    for (int i = threadIdx.x; i < 2 * TA * 8; i += blockDim.x) {
        const int h = i / (TA * 8);
        const int r = (i >> 3) % TA, c = i & 7;
        const int64_t row = tile * TA + r;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (row < M) {
            const uint2 b = *reinterpret_cast<const uint2*>(A + row * K + g * 128 + h * 64 + c * 8);
            i8x4_to_f16x4(b.x, o.x, o.y);
            i8x4_to_f16x4(b.y, o.z, o.w);
        }
        *reinterpret_cast<uint4*>(out + h * kAct + r * 128 + ((c ^ (r & 7)) << 4)) = o;
    }
    float* s = asc + static_cast<int64_t>(blockIdx.x) * (kAsc / 4);
    for (int i = threadIdx.x; i < GROUP * TA; i += blockDim.x) {
        // i = (((b * 4 + cq) * 2 + q) * 4 + m) * 4 + e: column quarter cq, chunk q of 16
        // columns, element e = 2 rl + c of thread m, i.e. activation row
        // 32 cq + 8 (2 q + rl) + 2 m + c
        const int b = i / TA, rem = i % TA;
        const int cq = rem / 32, q = (rem / 16) % 2, m = (rem / 4) % 4, e = rem % 4;
        const int r = 2 * q + e / 2, c = e % 2;
        const int64_t row = tile * TA + 32 * cq + 8 * r + 2 * m + c;
        s[i] = row < M ? AS[row * KB + g * GROUP + b] : 0.0f;
    }
}

// Zeroes C before a split-K contraction adds its partial tiles (a kernel, so
// that it takes part in the programmatic dependent launches).
__global__ void __launch_bounds__(256) zero_c_kernel(float* __restrict__ p, int64_t n) {
    pdl_wait();
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0.0f;
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

using TcwKernel = void (*)(CUtensorMap, CUtensorMap, TcwParams);

// The build of qdot_tcw_kernel for the weight format and the weight-scale
// layout with the most registers a thread that the device admits for 704
// threads in one block (the register file of an SM sub-partition holds six of
// the 22 warps), with its shared-memory size set; null if none.  Chosen once
// per device, format and layout.
template <bool Q5>
TcwKernel pick_kernel(int dev, bool rowmajor) {
    static std::mutex mu;
    static TcwKernel chosen[64][2] = {};
    static bool have[64][2] = {};
    if (dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    const int l = rowmajor ? 1 : 0;
    if (!have[dev][l]) {
        have[dev][l] = true;
        const TcwKernel cands[2][2] = {{qdot_tcw_kernel<80, false, Q5>, qdot_tcw_kernel<72, false, Q5>},
                                       {qdot_tcw_kernel<80, true, Q5>, qdot_tcw_kernel<72, true, Q5>}};
        for (TcwKernel k : cands[l]) {
            cudaFuncAttributes fa{};
            if (cudaFuncGetAttributes(&fa, k) != cudaSuccess || fa.maxThreadsPerBlock < kThreads) continue;
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) != cudaSuccess) continue;
            chosen[dev][l] = k;
            break;
        }
        cudaGetLastError();  // a declined candidate leaves no sticky error behind
    }
    return chosen[dev][l];
}

int g_skip = -1;
unsigned long long g_timeout = 4000000000ull;  // ~2 s at 2 GHz

}  // namespace

// Prompt shapes (M > 64) of qdot_t (q5: of q50_qdot_t, a.W holding Q5_0 blocks
// [N, K/32 * 20] bytes), block-scaled output only (the launch order:
// tile_act_kernel, the zeroing of C for split K, qdot_tcw_kernel).
// cudaErrorNotSupported when the shape or the operands do not suit this kernel
// (K % 128 != 0, weights or scale planes that TMA cannot load, not sm_103) or
// when the call may not allocate its activation workspace; the caller then
// takes the other tensor-core kernel.
cudaError_t launch_qdot_tcw(const QdotArgs& a, cudaStream_t stream, bool q5) {
    if (a.S != nullptr || a.no_alloc || a.M <= 64 || a.K % 128 != 0) return cudaErrorNotSupported;
    if (a.K > 0x7fffffffLL || a.M > 0x7fffffffLL || a.N > 0x7fffffffLL) return cudaErrorNotSupported;
    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorNotSupported;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3 || sms <= 0) return cudaErrorNotSupported;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(a.W) & 15u) != 0 || (reinterpret_cast<uintptr_t>(a.WS) & 15u) != 0)
        return cudaErrorNotSupported;
    const int64_t KB = a.K / 32;
    const bool rowmajor = a.ws_layout == PQ_WS_N_KB;
    if (!rowmajor && (a.N * 4) % 16 != 0) return cudaErrorNotSupported;

    TcwParams prm{};
    prm.C = a.C;
    prm.M = a.M;
    prm.N = a.N;
    prm.K = a.K;
    prm.ngroups = static_cast<int>(a.K / 128);
    prm.ws_rowmajor = rowmajor ? 1 : 0;
    prm.inject_skip_stage = g_skip;
    prm.timeout_cycles = g_timeout;
    const int64_t ta = (a.M + TA - 1) / TA;
    const int64_t tw = (a.N + TW - 1) / TW;
    const int64_t tiles = ta * tw;
    // K is split when the tiles are too few for the SMs: the smallest split
    // count whose units spread evenly (the busiest SM within ~5% of the mean),
    // each split keeping at least two scale groups
    int splits = 1;
    if (tiles < 4 * sms) {
        for (int s = 1; s <= std::max(1, prm.ngroups / 2); ++s) {
            const int64_t units = tiles * s;
            const double per_sm = static_cast<double>(units) / sms;
            const int64_t busiest = (units + sms - 1) / sms;
            splits = s;
            if (units >= sms && busiest <= per_sm * 1.05 + 1e-9) break;
        }
    }
    prm.groups_per_split = (prm.ngroups + splits - 1) / splits;
    splits = (prm.ngroups + prm.groups_per_split - 1) / prm.groups_per_split;
    if (tiles * splits > 0x7fffffffLL || ta * prm.ngroups > 0x7fffffffLL) return cudaErrorNotSupported;
    prm.splits = splits;
    prm.tiles_a = static_cast<int>(ta);
    prm.units = static_cast<int>(tiles * splits);
    prm.atomic = splits > 1 ? 1 : 0;

    CUtensorMap maps[2];
    {
        // int8 W [N, K]: box {128 bytes of K, 128 rows}, 128-byte swizzle; Q5_0 W [N, K/32 * 20]
        // bytes: box {80 bytes (one scale group), 128 rows}, no swizzle; zero fill past N
        const int64_t row_bytes = q5 ? KB * 20 : a.K;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(a.N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t box[2] = {q5 ? static_cast<cuuint32_t>(kQ5Row) : 128u, static_cast<cuuint32_t>(TW)};
        const cuuint32_t estr[2] = {1, 1};
        if (fn(&maps[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(a.W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, q5 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }
    {
        // WS: [N, KB] box {4 blocks, 128 rows}, or [KB, N] box {128 rows, 4 blocks}; zero fill past N
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(rowmajor ? KB : a.N),
                                    static_cast<cuuint64_t>(rowmajor ? a.N : KB)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>((rowmajor ? KB : a.N) * 4)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(rowmajor ? GROUP : TW),
                                   static_cast<cuuint32_t>(rowmajor ? TW : GROUP)};
        const cuuint32_t estr[2] = {1, 1};
        if (fn(&maps[1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(a.WS), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorNotSupported;
    }
    // the activation workspace of this stream: f16 stages, then the scales
    const size_t act_bytes = static_cast<size_t>(ta * prm.ngroups) * 2 * kAct;
    const size_t asc_bytes = static_cast<size_t>(ta * prm.ngroups) * kAsc;
    void* ws = nullptr;
    if (stream_workspace(stream, act_bytes + asc_bytes, &ws) != cudaSuccess) return cudaErrorNotSupported;
    prm.act = static_cast<const uint8_t*>(ws);
    prm.asc = static_cast<const uint8_t*>(ws) + act_bytes;
    cudaError_t e = launch_pdl(tile_act_kernel, dim3(static_cast<unsigned>(ta * prm.ngroups)), dim3(256), 0, stream,
                               a.A, a.AS, static_cast<uint8_t*>(ws),
                               reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + act_bytes), a.M, a.K);
    if (e != cudaSuccess) return e;
    if (prm.atomic) {
        const int64_t n = a.M * a.N;
        const int64_t blocks = std::min<int64_t>((n + 1023) / 1024, 2 * static_cast<int64_t>(sms));
        e = launch_pdl(zero_c_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, a.C, n);
        if (e != cudaSuccess) return e;
    }
    const int64_t grid = std::min<int64_t>(prm.units, sms);
    auto kern = q5 ? pick_kernel<true>(dev, rowmajor) : pick_kernel<false>(dev, rowmajor);
    if (!kern) return cudaErrorNotSupported;
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), static_cast<size_t>(kSmem), stream,
                      maps[0], maps[1], prm);
}

cudaError_t read_and_clear_status_w(unsigned* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_pq_status_w, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pq_status_w, &zero, sizeof(unsigned));
}

int tcw_kernel_regs() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const TcwKernel k = pick_kernel<false>(dev, true);
    if (!k) return 0;
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, k) == cudaSuccess ? fa.numRegs : 0;
}

void set_tcw_test_hooks(int inject_skip_group, unsigned long long timeout_cycles) {
    g_skip = inject_skip_group;
    g_timeout = timeout_cycles ? timeout_cycles : 4000000000ull;
}

}  // namespace pq
