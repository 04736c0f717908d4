// qdot_t for a few activation rows (1 <= M <= 64): warp-level MMA on weights
// streamed into shared memory by TMA.
//
// What it computes (the Q8_0 contraction of the qdot_t built-in, "the inner
// sum in integers, one scale multiply per block"):
//   C[m, n] = sum_b AS[m, b] * WS[n, b] * S_b[m, n],
//   S_b[m, n] = sum over the 32 k of block b of A[m, k] * W[n, k]   (exact integer).
//
// Why this design.  With M <= 64 the contraction is bound by the weight stream
// (N * K bytes).  A kernel whose computing warps load their own weight bytes
// keeps too few bytes in flight per SM to reach HBM bandwidth; here one
// producer warp per CTA keeps a ring of weight stages in flight by TMA while
// the consumer warps only compute.
//
// Work layout.
//   Cluster: KS CTAs (one per SM) that split K into chunks of whole 8-block
//   stages; the cluster owns a contiguous range of 8-row weight tiles and walks
//   it in passes of 128 rows.  Each CTA stages the activation rows of its K
//   chunk once, as f16 in shared memory, and keeps them for every pass.  After
//   a pass every lane sends its partial sums (st.async into distributed shared
//   memory, completing bytes on the receiver's mbarrier) to the CTA that
//   stores their share of C; that CTA sums them while the next pass computes
//   (two buffer halves by pass parity; a relaxed arrival tells the senders a
//   half has been read).  C is written once, with no zeroing pass and no
//   atomics, and no fence is on the path (a cluster-scope fence before a
//   remote arrival was measured at 3-4 thousand cycles a pass).
//   Stage: 128 weight rows x 256 bytes (eight Q8_0 blocks) in two TMA boxes of
//   128 rows x 128 bytes (the 128-byte swizzle span) and their f32 weight
//   scales in a third, on one mbarrier.  The TMA unit keeps few operations in
//   flight per SM, so the boxes are large: with four 32-row boxes and four
//   scale boxes per 16 KB stage the stream reached about a third of HBM
//   bandwidth.  A pass of fewer than 128 rows (the end of a cluster's range)
//   takes 32-row boxes instead, as few as cover its rows.  Eight blocks a
//   stage give each consumer warp several independent blocks between two
//   waits (a stage's time was measured to be one warp's dependency chain).
//   Consumer warp (box j, part kq): rows 32j .. 32j + 31 of the pass (four
//   n-tiles of 8) and 8 / KQ blocks of each stage, its m-tiles of 16 rows.
//   B fragments come from the stage by ldmatrix; A fragments and the
//   activation scales from the staged tile.
//
// Exactness.  A weight byte w is widened to the f16 value 1152 + w (w + 128
// placed under the f16 exponent of 1024: one xor and a byte permute per pair
// of bytes, exact), and the MMA's accumulator starts from -1152 * sum_k a_k,
// computed in the staging.  Every product a * (1152 + w) (|.| <= 128 * 1279)
// and every partial sum (|.| < 2^23) is an integer that f32 holds exactly, so
// each block sum comes out exact.
//
// K order inside a block.  ldmatrix gives lane q of a row group the bytes
// 4q .. 4q + 3 and 16 + 4q .. 16 + 4q + 3 of the block; MMA step 0 takes the
// first four (as K positions 2q, 2q + 1, 2q + 8, 2q + 9), step 1 the second.
// The staged activation tile keeps, per row and block, the same eight
// elements of lane q in one 16-byte piece, so each block sum covers the
// block's 32 k once.
//
// Safety.  Every mbarrier wait is bounded (a clock64 limit).  A wait that
// gives up sets this file's device status word and a CTA-wide abort flag;
// every role then runs out its loops without waiting or working, TMA loads in
// flight are drained with bounded waits, and every thread of every CTA meets
// at one last cluster barrier (after waiting, bounded, for the other CTAs'
// last arrivals on its barriers), so no CTA leaves while another may still
// write to its shared memory.  No trap, no unbounded spin.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pq_device.cuh"
#include "pq_internal.h"
#include "tc_ptx.cuh"

namespace pq {

// Nonzero after a bounded wait of this file's kernel gave up.
__device__ unsigned g_pq_status_mmt;

namespace {

constexpr int kBoxRows = 32;                          // weight rows per TMA box: one consumer warp's rows
constexpr int kBoxes = 4;                             // boxes per stage
constexpr int kPassRows = kBoxRows * kBoxes;          // 128 weight rows per pass
constexpr int kPassTiles = kPassRows / 8;             // 8-row tiles per pass
constexpr int kHalves = 2;                            // 128-byte column groups per stage (128B swizzle span)
constexpr int kStageBlocks = 4 * kHalves;             // Q8_0 blocks per stage (256 bytes of a row)
constexpr int kW8Box = kBoxRows * 128;                // 4 KB: 32 rows of one column group
constexpr int kW8Half = kBoxes * kW8Box;              // 16 KB: the pass's rows in one column group
constexpr int kW8 = kHalves * kW8Half;                // 32 KB of weight bytes per stage
constexpr int kWSBox = kBoxRows * kStageBlocks * 4;   // 1 KB of weight scales per 32 rows
constexpr int kWS = kBoxes * kWSBox;
constexpr int kMaxStages = 8;
constexpr int kMaxCluster = 8;
constexpr int kSmemLimit = 227 * 1024;
constexpr float kBias = 1152.0f;                      // 1024 + 128

// Consumer warps: kBoxes x KQ (K parts of a stage) x MG (groups of m-tiles).
// The register file of an SM sub-partition (16384 registers) bounds a thread
// by the warps that land on one sub-partition: 9 warps (8 consumers and the
// producer) put 3 on one and allow 168 registers, which two m-tiles per warp
// need without spilling (four m-tiles go to two warp groups of two).  Each
// consumer warp reads every weight-scale row of its blocks at once and the
// staged activation fragments of its blocks, so fewer K parts mean fewer
// shared-memory wavefronts per stage.
template <int MT>
struct MmtCfg {
    // one m-tile: 2 K parts (measured at M = 16, K = 4096, N = 11008: 21.5 us
    // against 23.6 with 4 and 27 with 1; fewer parts also shrink the partials'
    // buffer, leaving room for a deeper ring)
    static constexpr int KQ = MT <= 2 ? 2 : 1;  // consumer warps per box and m-group (4 or 8 blocks each)
    static constexpr int MG = MT == 4 ? 2 : 1;        // m-groups
    static constexpr int MTW = MT / MG;               // m-tiles per consumer warp
    static constexpr int BPW = kStageBlocks / KQ;     // blocks per consumer warp and stage
    static constexpr int NC = kBoxes * KQ * MG;       // consumer warps
    static constexpr int kThreads = 32 * (NC + 1);    // + the producer warp
    static constexpr int R = 16 * MT;                 // staged activation rows (zero past M)
    static constexpr int kSlots = kBoxes * MT * 4 * 32;  // float4 partials per quarter
    static constexpr int kRed = 2 * KQ * kSlots * 16;  // received partials, two halves (pass parity)
};

struct MmtParams {
    const int8_t* A;    // [M, K]
    const float* AS;    // [M, K/32]
    float* C;           // [M, N]
    int64_t M, N, K;
    int KB;
    int nbc;            // blocks per K chunk (a multiple of kStageBlocks)
    int ntiles;         // 8-row weight tiles, ceil(N / 8)
    int clusters;
    int stages;         // ring depth
    int ws_layout;      // 0: WS [N, K/32]; 1: WS [K/32, N]
    int vec2;           // C 8-byte aligned and N even: float2 stores
    int inject_skip;    // test hook: the producer never fills this stage (-1: off)
    int early_weights;  // W / WS may be read before griddepcontrol.wait (QdotArgs::early_weights)
    unsigned long long timeout_cycles;
    uint32_t off_ws, off_a, off_asc, off_red, off_bar;  // shared-memory regions
    uint32_t a_rs;      // bytes per row of the staged activation tile (nbc * 64 + 64)
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// The cluster barrier, in halves: every thread of every CTA arrives
// (barrier.cluster.arrive.relaxed, inline), then waits (threads may arrive
// apart; a thread waits before it arrives again).
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }

// One arrival on the mbarrier at shared-memory offset `bar` in CTA `cta` of
// the cluster.  Relaxed: it tells the other CTA that this one has read a
// buffer, and those reads have returned their values before it is issued.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t cta) {
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
        "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [ra];\n\t}"
        ::"r"(bar), "r"(cta) : "memory");
}

// 16 bytes into the shared memory of CTA `cta` at offset `addr`, completing
// 16 bytes of transaction on that CTA's mbarrier at offset `bar`.
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint32_t bar, uint32_t cta, const uint4& v) {
    asm volatile(
        "{\n\t.reg .b32 ra, rb;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %2;\n\t"
        "mapa.shared::cluster.u32 rb, %1, %2;\n\t"
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [ra], {%3, %4, %5, %6}, [rb];\n\t}"
        ::"r"(addr), "r"(bar), "r"(cta), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
// Non-blocking test at cluster scope (the waits on other CTAs' arrivals poll:
// a suspended try_wait was measured to notice remote arrivals late).
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& d0, uint32_t& d1, uint32_t& d2, uint32_t& d3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d0), "=r"(d1), "=r"(d2), "=r"(d3) : "r"(addr));
}
// N consecutive floats (N = 1, 2 or 4) from shared memory.
template <int N>
__device__ __forceinline__ void lds_vec(uint32_t addr, float (&r)[N]) {
    if constexpr (N == 4) {
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]) : "r"(addr));
    } else if constexpr (N == 2) {
        asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(r[0]), "=f"(r[1]) : "r"(addr));
    } else {
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r[0]) : "r"(addr));
    }
}
__device__ __forceinline__ uint64_t lds64(uint32_t addr) {
    uint64_t v;
    asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(addr));
    return v;
}

// D += A * B on one m16n8k16 tile: A 16 x 16 f16 (row), B 16 x 8 f16 (column), D f32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + C on one m16n8k16 tile, C in registers of its own.
__device__ __forceinline__ void mma_16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1, const float4& c) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y), "f"(c.z), "f"(c.w));
}

// Four weight bytes -> two f16x2 of 1152 + w (bytes 0, 1 in lo; 2, 3 in hi).
__device__ __forceinline__ void w8x4_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x4140u);
    hi = __byte_perm(u, 0x64646464u, 0x4342u);
}

// ------------------------------------------------------------ bounded waits

// The CTA's abort flag, a word of shared memory at shared-window address a.
__device__ __forceinline__ uint32_t abort_get(uint32_t a) {
    uint32_t v;
    asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void set_abort(uint32_t a) {
    if (abort_get(a) == 0) {
        asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(a), "r"(1u) : "memory");
        atomicOr(&g_pq_status_mmt, 1u);
    }
}

// Waits for the phase of `bar` with the given parity (CTA or cluster scope):
// true once it has completed; false if it has not and the CTA is aborting, or
// the wait ran past its limit (which starts the abort).
template <bool CLUSTER>
__device__ __forceinline__ bool bounded_wait(uint64_t* bar, uint32_t parity, uint32_t abort_a,
                                             unsigned long long limit) {
    auto test = [&] {
        return CLUSTER ? mbar_test_wait_cluster(tc::smem_u32(bar), parity) : tc::mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    if (abort_get(abort_a)) return false;
    const long long t0 = clock64();
    for (uint32_t n = 1;; ++n) {
        if (test()) return true;
        if ((n & 15) == 0) {
            if (abort_get(abort_a)) return false;
            if (static_cast<unsigned long long>(clock64() - t0) > limit) {
                set_abort(abort_a);
                return false;
            }
        }
    }
}

// Drain wait for TMA loads already issued: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit) {
    const long long t0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
        if (static_cast<unsigned long long>(clock64() - t0) > limit) {
            atomicOr(&g_pq_status_mmt, 2u);
            return;
        }
    }
}

// ------------------------------------------------------------ staging

// Thread qq's piece of activation row r, local block b (bytes 4qq .. 4qq + 3
// in v0, 16 + 4qq .. 16 + 4qq + 3 in v1; scale d; the block's byte sum over
// the four pieces) into the staged tile: the f16 elements at [r][b][qq]
// (rows a_rs bytes apart), and from pieces 0 and 1 the block's record of
// scale pairs and MMA starting values -1152 * sum.
template <int MT>
__device__ __forceinline__ void stage_piece(uint8_t* smem, const MmtParams& p, int r, int b, int qq, uint32_t v0,
                                            uint32_t v1, float d, int sum) {
    uint4 o;
    i8x4_to_f16x4(v0, o.x, o.y);
    i8x4_to_f16x4(v1, o.z, o.w);
    *reinterpret_cast<uint4*>(smem + p.off_a + static_cast<uint32_t>(r) * p.a_rs + b * 64 + 16 * qq) = o;
    // record (b, m-tile, row of the 8-row group): {d(g), d(g), d(g+8), d(g+8), c(g), c(g), c(g+8), c(g+8)}
    if (qq < 2) {
        float* rec = reinterpret_cast<float*>(smem + p.off_asc +
                                              ((static_cast<uint32_t>(b) * MT + (r >> 4)) * 8 + (r & 7)) * 32);
        const float val = qq == 0 ? d : -kBias * static_cast<float>(sum);
        *reinterpret_cast<float2*>(rec + 4 * qq + 2 * ((r >> 3) & 1)) = make_float2(val, val);
    }
}

// ------------------------------------------------------------ kernel

template <int MT>
__global__ void __launch_bounds__(MmtCfg<MT>::kThreads, 1)
    qdot_mmt_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap smap,
                    const __grid_constant__ CUtensorMap wmap32, const __grid_constant__ CUtensorMap smap32,
                    const MmtParams p) {
    using CF = MmtCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t ks = cluster_size();  // a power of two <= 8
    const int ci = static_cast<int>(blockIdx.x / ks);
    const int S = p.stages;
    // the cluster's 8-row tiles [t0, t1), walked in passes of kPassTiles
    const int t0 = static_cast<int>(static_cast<int64_t>(ci) * p.ntiles / p.clusters);
    const int t1 = static_cast<int>(static_cast<int64_t>(ci + 1) * p.ntiles / p.clusters);
    const int npass = (t1 - t0 + kPassTiles - 1) / kPassTiles;
    const int64_t row_end = min(static_cast<int64_t>(t1) * 8, p.N);
    // this CTA's K chunk: blocks [b0, b0 + nbr), in nst stages
    const int b0 = static_cast<int>(rank) * p.nbc;
    const int nbr = max(0, min(p.nbc, p.KB - b0));
    const int nst = (nbr + kStageBlocks - 1) / kStageBlocks;

    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    uint64_t* empty = full + S;
    uint64_t* ready = empty + S;  // [2]: the partials of a pass have all arrived here (by parity of the pass)
    uint64_t* done = ready + 2;   // [2]: every CTA has read the partials this one sent it
    const uint32_t abort_flag = tc::smem_u32(done + 2);
    const unsigned long long limit = p.timeout_cycles;

    // The producer sets up the ring and starts streaming at once; the
    // consumers meet it on named barrier 2 before their first wait on the
    // ring.  The cluster's barriers (ready / done) are initialised by consumer
    // thread 0; every thread arrives on the cluster barrier now and waits just
    // before its first remote operation (the end of the first pass).
    if (warp == CF::NC) {
        if (lane == 0) {
            for (int s = 0; s < S; ++s) {
                tc::mbar_init(&full[s], 1);
                tc::mbar_init(&empty[s], CF::NC);
            }
            asm volatile("st.volatile.shared.u32 [%0], %1;" ::"r"(abort_flag), "r"(0u) : "memory");
            tc::fence_mbar_init();
        }
        __syncwarp();
        asm volatile("bar.arrive 2, %0;" ::"r"(CF::kThreads) : "memory");
    } else {
        if (tid == 0) {
            for (int b = 0; b < 2; ++b) {
                tc::mbar_init(&ready[b], 1);  // the owner's expect_tx; the bytes come from the cluster
                tc::mbar_init(&done[b], ks);
            }
            tc::fence_mbar_init();
        }
        tc::named_bar_sync(2, CF::kThreads);
    }
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");

    const int total = npass * nst;  // stages this CTA consumes
    if (warp == CF::NC) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            auto coords = [&](int it, int& x, int& y, int& nbox) {
                const int pass = it / nst, s = it - pass * nst;
                const int tile0 = t0 + pass * kPassTiles;
                y = tile0 * 8;
                nbox = min(kBoxes, ((t1 - tile0) * 8 + kBoxRows - 1) / kBoxRows);
                x = b0 + s * kStageBlocks;
            };
            // Before waiting on the preceding kernel: with early_weights (the
            // preceding kernel is the library's quantizer, which let this one in
            // only once every kernel before it had completed) the first stages
            // are loaded; otherwise L2 is asked for them (a hint that cannot
            // return stale data; the loads come after the wait).
            const int first = min(S, total);
            if (!p.early_weights) {
                for (int it = 0; it < first; ++it) {
                    int x, y, nbox;
                    coords(it, x, y, nbox);
                    for (int h = 0; h < kHalves; ++h) {
                        if (nbox == kBoxes) tc::tma_prefetch_2d(&wmap, x * 32 + h * 128, y);
                        else for (int i = 0; i < nbox; ++i) tc::tma_prefetch_2d(&wmap32, x * 32 + h * 128, y + i * kBoxRows);
                    }
                }
                pdl_wait();
            }
            int it = 0, slot = 0;
            uint32_t phase = 0;  // (it / S) & 1
            for (; it < total; ++it, slot = slot + 1 == S ? 0 : slot + 1, phase ^= slot == 0 ? 1u : 0u) {
                if (p.early_weights && it == first) pdl_wait();
                if (it >= S && (abort_get(abort_flag) || !bounded_wait<false>(&empty[slot], phase ^ 1, abort_flag, limit)))
                    break;
                if (it == p.inject_skip) continue;
                int x, y, nbox;
                coords(it, x, y, nbox);
                tc::mbar_arrive_expect_tx(&full[slot],
                                          static_cast<uint32_t>(nbox * (kHalves * kW8Box + kWSBox)));
                uint8_t* wdst = smem + slot * kW8;
                uint8_t* sdst = smem + p.off_ws + slot * kWS;
                if (nbox == kBoxes) {
                    // a whole pass: boxes of 128 rows
                    for (int h = 0; h < kHalves; ++h)
                        tc::tma_load_2d(wdst + h * kW8Half, &wmap, &full[slot], x * 32 + h * 128, y);
                    if (p.ws_layout == 0) tc::tma_load_2d(sdst, &smap, &full[slot], x, y);
                    else tc::tma_load_2d(sdst, &smap, &full[slot], y, x);
                } else {
                    for (int i = 0; i < nbox; ++i) {
                        for (int h = 0; h < kHalves; ++h)
                            tc::tma_load_2d(wdst + h * kW8Half + i * kW8Box, &wmap32, &full[slot], x * 32 + h * 128,
                                            y + i * kBoxRows);
                        if (p.ws_layout == 0)
                            tc::tma_load_2d(sdst + i * kWSBox, &smap32, &full[slot], x, y + i * kBoxRows);
                        else tc::tma_load_2d(sdst + i * kWSBox, &smap32, &full[slot], y + i * kBoxRows, x);
                    }
                }
            }
            if (p.early_weights && it <= first) pdl_wait();  // (no stage past the first ring, or an early end)
            // loads still in flight land before the CTA may exit
            for (int j = max(0, it - S); j < it; ++j)
                if (j != p.inject_skip) drain_wait(&full[j % S], (j / S) & 1, limit);
        }
        cluster_wait();
    } else {
        // ---------------------------------------------------------- consumers
        const int ctid = tid;  // consumer threads are 0 .. NC * 32 - 1
        constexpr int NCT = CF::NC * 32;
        pdl_wait();
        // staging: the chunk's activation rows (zero past M and past the chunk),
        // four threads per block (thread q: bytes 4q .. 4q + 3 and 16 + 4q ..
        // 16 + 4q + 3, the lane's piece of the staged row), consecutive
        // threads on consecutive pieces of one row (coalesced loads,
        // conflict-free stores); each thread issues the loads of kBatch pieces
        // before using them
        constexpr int kBatch = 8;
        const int nunits = CF::R * p.nbc * 4;
        for (int base = 0; base < nunits; base += kBatch * NCT) {
            uint32_t v0[kBatch], v1[kBatch];
            float d[kBatch];
            bool live[kBatch];
#pragma unroll
            for (int h = 0; h < kBatch; ++h) {
                const int i = base + h * NCT + ctid;
                const int qq = i & 3, rb = i >> 2;
                const int r = rb / p.nbc, b = rb - r * p.nbc;
                live[h] = i < nunits && r < p.M && b < nbr;
                v0[h] = v1[h] = 0u;
                d[h] = 0.0f;
                if (live[h]) {
                    const int8_t* src = p.A + r * p.K + static_cast<int64_t>(b0 + b) * 32 + 4 * qq;
                    v0[h] = *reinterpret_cast<const uint32_t*>(src);
                    v1[h] = *reinterpret_cast<const uint32_t*>(src + 16);
                    d[h] = p.AS[r * static_cast<int64_t>(p.KB) + b0 + b];
                }
            }
#pragma unroll
            for (int h = 0; h < kBatch; ++h) {
                const int i = base + h * NCT + ctid;
                const int qq = i & 3, rb = i >> 2;
                const int r = rb / p.nbc, b = rb - r * p.nbc;
                int sum = __dp4a(static_cast<int>(v0[h]), 0x01010101, __dp4a(static_cast<int>(v1[h]), 0x01010101, 0));
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (i < nunits) stage_piece<MT>(smem, p, r, b, qq, v0[h], v1[h], d[h], sum);
            }
        }
        tc::named_bar_sync(1, NCT);
        pdl_trigger();

        const int j = warp & (kBoxes - 1), kq = (warp / kBoxes) % CF::KQ, mh = warp / (kBoxes * CF::KQ);
        const int g = lane >> 2, q = lane & 3;
        const uint32_t sbase = tc::smem_u32(smem);
        // ldmatrix row addresses within a box: matrix mi = lane / 8 is n-tile
        // 2h + mi / 2, 16-byte chunk 2u + mi % 2 of the block, row lane % 8
        // (chunk c of row r sits at chunk c ^ (r % 8): the 128-byte swizzle)
        uint32_t ldm_off[CF::BPW][2];
#pragma unroll
        for (int ub = 0; ub < CF::BPW; ++ub) {
            const int u = kq * CF::BPW + ub;  // block of the stage: column group u / 4, block u % 4 in it
            const int mi = lane >> 3, i = lane & 7;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                ldm_off[ub][h] = (u >> 2) * kW8Half + (8 * (2 * h + (mi >> 1)) + i) * 128 +
                                 (((2 * (u & 3) + (mi & 1)) ^ i) << 4);
        }
        const uint32_t a_lane = sbase + p.off_a + g * p.a_rs + q * 16;
        const uint32_t asc_lane = sbase + p.off_asc + g * 32;
        // partials of a pass, in the CTA that stores them: slot sl of the pass
        // tile goes to CTA sl % ks, at [source CTA][quarter kq][sl / ks], in the
        // half of the buffer of the pass's parity
        const int share = CF::kSlots / static_cast<int>(ks);
        const uint32_t red_half = static_cast<uint32_t>(CF::KQ * CF::kSlots * 16);
        const uint32_t red_base = sbase + p.off_red;
        const uint32_t ready_a = tc::smem_u32(ready), done_a = tc::smem_u32(done);

        // the owner's side of pass pp: wait for the cluster's partials, sum, store
        auto reduce = [&](int pp) {
            const int b = pp & 1;
            if (ctid == 0 && abort_get(abort_flag) == 0)
                tc::mbar_arrive_expect_tx(&ready[b], static_cast<uint32_t>(ks * CF::KQ * share * 16));
            const bool ok = bounded_wait<true>(&ready[b], (pp >> 1) & 1, abort_flag, limit);
            if (ok) {
                const int tile0 = t0 + pp * kPassTiles;
                const int nrows = min(kPassRows, (t1 - tile0) * 8);
                for (int si = ctid; si < share; si += NCT) {
                    const int sl = si * static_cast<int>(ks) + static_cast<int>(rank);
                    const int jj = (sl >> 7) / MT;
                    if (jj * kBoxRows >= nrows) continue;  // a box past the pass's rows
                    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                    for (uint32_t src = 0; src < ks; ++src)
#pragma unroll
                        for (int h = 0; h < CF::KQ; ++h) {
                            const float4 o = tc::lds128f(red_base + b * red_half +
                                                         ((src * CF::KQ + h) * share + si) * 16);
                            v.x += o.x;
                            v.y += o.y;
                            v.z += o.z;
                            v.w += o.w;
                        }
                    const int ln = sl & 31, t = (sl >> 5) & 3, mt = (sl >> 7) % MT;
                    const int64_t m = 16 * mt + (ln >> 2);
                    const int64_t n = static_cast<int64_t>(tile0) * 8 + jj * kBoxRows + 8 * t + 2 * (ln & 3);
                    if (n + 1 < row_end && p.vec2) {
                        if (m < p.M) *reinterpret_cast<float2*>(p.C + m * p.N + n) = make_float2(v.x, v.y);
                        if (m + 8 < p.M) *reinterpret_cast<float2*>(p.C + (m + 8) * p.N + n) = make_float2(v.z, v.w);
                    } else {
                        if (n < row_end) {
                            if (m < p.M) p.C[m * p.N + n] = v.x;
                            if (m + 8 < p.M) p.C[(m + 8) * p.N + n] = v.z;
                        }
                        if (n + 1 < row_end) {
                            if (m < p.M) p.C[m * p.N + n + 1] = v.y;
                            if (m + 8 < p.M) p.C[(m + 8) * p.N + n + 1] = v.w;
                        }
                    }
                }
            }
            tc::named_bar_sync(1, NCT);
            // the senders may reuse this half of the buffer
            if (ctid == 0 && ok && abort_get(abort_flag) == 0)
                for (uint32_t c = 0; c < ks; ++c) mbar_arrive_remote(done_a + b * 8, c);
        };

        int slot = 0;
        uint32_t phase = 0;  // (stage counter / S) & 1
        for (int pass = 0; pass <= npass; ++pass) {
            if (pass < npass) {
                const int tile0 = t0 + pass * kPassTiles;
                const int nrows = min(kPassRows, (t1 - tile0) * 8);
                const bool active = j * kBoxRows < nrows;
                // weight scales of the stage: [128 rows][4 blocks] for WS [N, K/32]
                // (one box or four stacked); for WS [K/32, N] [4 blocks][128 rows]
                // in a whole pass, [box][4 blocks][32 rows] otherwise
                const bool whole = nrows == kPassRows;
                const uint32_t ws_j = (p.ws_layout == 1 && whole) ? kBoxRows * 4 : kWSBox;
                const uint32_t ws_u = whole ? kPassRows * 4 : kBoxRows * 4;
                uint64_t acc[CF::MTW][4][2];  // m-tiles mh * MTW + mw
#pragma unroll
                for (int mt = 0; mt < CF::MTW; ++mt)
#pragma unroll
                    for (int t = 0; t < 4; ++t) acc[mt][t][0] = acc[mt][t][1] = 0ull;

                for (int s = 0; s < nst; ++s) {
                    const bool ok = __all_sync(0xffffffffu, bounded_wait<false>(&full[slot], phase, abort_flag, limit));
                    if (ok && active) {
                        const uint32_t wbox = sbase + slot * kW8 + j * kW8Box;
                        const uint32_t sbox = sbase + p.off_ws + slot * kWS + j * ws_j;
                        // weight scales of rows 8t + 2q, 8t + 2q + 1 for each of the
                        // warp's blocks.  One m-tile: all blocks at once (with WS
                        // [N, K/32] a row's blocks are adjacent: one load of BPW
                        // floats per row); more m-tiles (whose registers are
                        // scarcer and whose loads serve two m-tiles): per block.
                        constexpr bool kWsAll = MT == 1;
                        uint64_t ws2[kWsAll ? CF::BPW : 1][4];
                        auto load_ws = [&](int ub, uint64_t (&dst)[4]) {
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                if (p.ws_layout == 1) {
                                    dst[t] = lds64(sbox + (kq * CF::BPW + ub) * ws_u + (8 * t + 2 * q) * 4);
                                } else {
                                    const uint32_t a = sbox + ((8 * t + 2 * q) * kStageBlocks + kq * CF::BPW + ub) * 4;
                                    dst[t] = f2_pack(tc::lds32(a), tc::lds32(a + kStageBlocks * 4));
                                }
                            }
                        };
                        if constexpr (kWsAll) {
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                if (p.ws_layout == 1) {
#pragma unroll
                                    for (int ub = 0; ub < CF::BPW; ++ub)
                                        ws2[ub][t] = lds64(sbox + (kq * CF::BPW + ub) * ws_u + (8 * t + 2 * q) * 4);
                                } else {
                                    const uint32_t a = sbox + ((8 * t + 2 * q) * kStageBlocks + kq * CF::BPW) * 4;
                                    float r0[CF::BPW], r1[CF::BPW];
                                    lds_vec<CF::BPW>(a, r0);
                                    lds_vec<CF::BPW>(a + kStageBlocks * 4, r1);
#pragma unroll
                                    for (int ub = 0; ub < CF::BPW; ++ub)
                                        ws2[ub][t] = f2_pack(__float_as_uint(r0[ub]), __float_as_uint(r1[ub]));
                                }
                            }
                        }
#pragma unroll
                        for (int ub = 0; ub < CF::BPW; ++ub) {
                            const int u = kq * CF::BPW + ub;
                            const int bl = s * kStageBlocks + u;  // block within the chunk
                            uint32_t d8[4][2];
                            ldmatrix_x4(wbox + ldm_off[ub][0], d8[0][0], d8[0][1], d8[1][0], d8[1][1]);
                            ldmatrix_x4(wbox + ldm_off[ub][1], d8[2][0], d8[2][1], d8[3][0], d8[3][1]);
                            if constexpr (!kWsAll) load_ws(ub, ws2[0]);
                            const uint64_t (&wsb)[4] = ws2[kWsAll ? ub : 0];
                            uint32_t bf[4][4];
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                w8x4_biased(d8[t][0], bf[t][0], bf[t][1]);
                                w8x4_biased(d8[t][1], bf[t][2], bf[t][3]);
                            }
#pragma unroll
                            for (int mw = 0; mw < CF::MTW; ++mw) {
                                const int mt = mh * CF::MTW + mw;
                                const uint32_t ar = a_lane + 16 * mt * p.a_rs + bl * 64;
                                const uint4 lo = tc::lds128(ar);                // row g
                                const uint4 hi = tc::lds128(ar + 8 * p.a_rs);   // row g + 8
                                const uint32_t rr = asc_lane + (bl * MT + mt) * 8 * 32;
                                const uint4 sc = tc::lds128(rr);         // d(g), d(g), d(g+8), d(g+8)
                                const float4 c0 = tc::lds128f(rr + 16);  // starting values
                                const uint64_t dg = f2_pack(sc.x, sc.y), dg8 = f2_pack(sc.z, sc.w);
#pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    float sv[4];
                                    mma_16816_c(sv, lo.x, hi.x, lo.y, hi.y, bf[t][0], bf[t][1], c0);
                                    mma_16816(sv, lo.z, hi.z, lo.w, hi.w, bf[t][2], bf[t][3]);
                                    acc[mw][t][0] = f2_fma(f2_mul(dg, wsb[t]),
                                                           f2_pack(__float_as_uint(sv[0]), __float_as_uint(sv[1])),
                                                           acc[mw][t][0]);
                                    acc[mw][t][1] = f2_fma(f2_mul(dg8, wsb[t]),
                                                           f2_pack(__float_as_uint(sv[2]), __float_as_uint(sv[3])),
                                                           acc[mw][t][1]);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&empty[slot]);
                    if (++slot == S) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }

                // send this pass's partials to the CTAs that store them; the
                // half of the buffer is free once they have read pass - 2
                if (pass == 0) cluster_wait();
                const int b = pass & 1;
                const bool ok = pass < 2 ? abort_get(abort_flag) == 0
                                         : bounded_wait<true>(&done[b], ((pass - 2) >> 1) & 1, abort_flag, limit);
                if (ok) {
                    const uint32_t owner = static_cast<uint32_t>(lane) & (ks - 1);  // slot % ks (ks divides 32)
#pragma unroll
                    for (int mw = 0; mw < CF::MTW; ++mw)
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int sl = ((j * MT + mh * CF::MTW + mw) * 4 + t) * 32 + lane;
                            const uint32_t dst = red_base + b * red_half +
                                                 ((rank * CF::KQ + kq) * share + sl / static_cast<int>(ks)) * 16;
                            st_async_v4(dst, ready_a + b * 8, owner,
                                        make_uint4(static_cast<uint32_t>(acc[mw][t][0]),
                                                   static_cast<uint32_t>(acc[mw][t][0] >> 32),
                                                   static_cast<uint32_t>(acc[mw][t][1]),
                                                   static_cast<uint32_t>(acc[mw][t][1] >> 32)));
                        }
                }
            } else if (npass == 0) {
                cluster_wait();
            }
            // the previous pass's share of C, while this pass's partials travel
            if (pass >= 1) reduce(pass - 1);
        }
        // every CTA has read what this one sent in the last two passes, so no
        // arrival on this CTA's barriers is still on its way
        for (int pp = max(0, npass - 2); pp < npass; ++pp)
            (void)bounded_wait<true>(&done[pp & 1], (pp >> 1) & 1, abort_flag, limit);
    }
    // no CTA leaves while another may still write to its shared memory
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
    cluster_wait();
}

// ------------------------------------------------------------ host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D map of a row-major plane [outer, inner] of `esize`-byte elements, box
// {box_inner, box_outer}, zero fill outside the plane.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t inner, int64_t outer,
              int64_t esize, int box_inner, int box_outer, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner * esize)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Layout {
    int stages = 0;
    uint32_t off_ws = 0, off_a = 0, off_asc = 0, off_red = 0, off_bar = 0, bytes = 0;
};

// Shared-memory layout for a K chunk of nbc blocks with the deepest ring that
// fits (0 stages: nothing fits).
template <int MT>
Layout layout_for(int nbc) {
    using CF = MmtCfg<MT>;
    Layout L;
    const int64_t a_rs = static_cast<int64_t>(nbc) * 64 + 64;  // = 64 mod 128: conflict-free row pairs
    const int64_t fixed = CF::R * a_rs + static_cast<int64_t>(nbc) * MT * 256 + CF::kRed;
    for (int s = kMaxStages; s >= 2; --s) {
        const int64_t bytes = static_cast<int64_t>(s) * (kW8 + kWS) + fixed + (2 * s + 4) * 8 + 16 + 1024;
        if (bytes <= kSmemLimit) {
            L.stages = s;
            L.off_ws = static_cast<uint32_t>(s * kW8);
            L.off_a = L.off_ws + static_cast<uint32_t>(s * kWS);
            L.off_asc = L.off_a + static_cast<uint32_t>(CF::R * a_rs);
            L.off_red = L.off_asc + static_cast<uint32_t>(nbc * MT * 256);
            L.off_bar = L.off_red + static_cast<uint32_t>(CF::kRed);
            L.bytes = static_cast<uint32_t>(bytes);
            return L;
        }
    }
    return L;
}

int g_skip_stage = -1;
unsigned long long g_timeout = 4000000000ull;  // ~2 s at 2 GHz
int g_small_kernel = 1;                        // 1: this kernel where it applies; 0: the register-fed one
int g_force_ks = 0;                            // test hook: only this cluster size (0: the cost model's choice)
std::atomic<int> g_last_cfg[4];                // the last launch's cluster size, clusters, ring stages, K chunk

struct Choice {
    int ks = 0, clusters = 0, nbc = 0;
    Layout L;
};

template <int MT>
cudaError_t launch_mt(const CUtensorMap* maps, MmtParams p, cudaStream_t stream) {
    using CF = MmtCfg<MT>;
    auto kern = qdot_mmt_kernel<MT>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
    // per device: SM count (0: not sm_103), shared-memory limit raised
    static std::mutex dmu;
    static int dev_sms[64];
    static bool dev_have[64];
    int sms = 0;
    {
        std::lock_guard<std::mutex> lk(dmu);
        if (!dev_have[dev]) {
            int n = 0, major = 0, minor = 0;
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
            if (major == 10 && minor == 3 && n > 0) {
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
                if (e != cudaSuccess) return e;
                dev_sms[dev] = n;
            }
            dev_have[dev] = true;
        }
        sms = dev_sms[dev];
    }
    if (sms <= 0) return cudaErrorNotSupported;

    // K split: for each cluster size the chunk (whole stages), the ring that
    // fits and how many clusters the device runs at once; take the one whose
    // busiest CTA the time model below puts first
    Choice best;
    int64_t best_cost = -1;
    for (int ks : {8, 4, 2, 1}) {
        if (g_force_ks != 0 && ks != g_force_ks) continue;
        const int nbc = (p.KB + ks - 1) / ks;
        const int chunk = (nbc + kStageBlocks - 1) / kStageBlocks * kStageBlocks;
        const int kse = (p.KB + chunk - 1) / chunk;
        if ((kse & (kse - 1)) != 0) continue;  // the partials' owner is lane % ks: a power of two
        if (g_force_ks != 0 && kse != g_force_ks) continue;
        const Layout L = layout_for<MT>(chunk);
        if (L.stages < 2) continue;
        static std::mutex mu;
        static int cache[64][4][kMaxCluster + 1];  // [device][MT index][ks] -> clusters + 1 (0: unknown)
        const int mti = MT == 1 ? 0 : MT == 2 ? 1 : 2;
        int nclu = 0;
        {
            std::lock_guard<std::mutex> lk(mu);
            if (dev < 64 && cache[dev][mti][kse] > 0) nclu = cache[dev][mti][kse] - 1;
            else {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(static_cast<unsigned>(kse * (sms / kse)));
                cfg.blockDim = dim3(CF::kThreads);
                cfg.dynamicSmemBytes = kSmemLimit;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = static_cast<unsigned>(kse);
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&nclu, kern, &cfg) != cudaSuccess) {
                    (void)cudaGetLastError();
                    nclu = 0;
                }
                if (dev < 64) cache[dev][mti][kse] = nclu + 1;
            }
        }
        if (nclu <= 0) continue;
        nclu = static_cast<int>(std::min<int64_t>(nclu, p.ntiles));
        // time of the busiest CTA: its stages, each taking the longer of its
        // bytes at an SM's share of HBM bandwidth (~23 B/cycle) and the load
        // latency under load (~3500 cycles) over the ring depth
        const int64_t tiles = (p.ntiles + nclu - 1) / nclu;
        const int64_t whole = tiles / kPassTiles, tail = tiles % kPassTiles;
        const int64_t nstage = chunk / kStageBlocks;
        const int64_t t_lat = 3500 / L.stages;
        const int64_t t_whole = std::max<int64_t>((kW8 + kWS) / 23, t_lat);
        const int64_t t_tail =
            std::max<int64_t>((tail * 8 + kBoxRows - 1) / kBoxRows * (kHalves * kW8Box + kWSBox) / 23, t_lat);
        const int64_t cost = nstage * (whole * t_whole + (tail ? t_tail : 0));
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.ks = kse;
            best.clusters = nclu;
            best.nbc = chunk;
            best.L = L;
        }
    }
    if (best_cost < 0) return cudaErrorNotSupported;

    g_last_cfg[0].store(best.ks, std::memory_order_relaxed);
    g_last_cfg[1].store(best.clusters, std::memory_order_relaxed);
    g_last_cfg[2].store(best.L.stages, std::memory_order_relaxed);
    g_last_cfg[3].store(best.nbc, std::memory_order_relaxed);
    p.nbc = best.nbc;
    p.clusters = best.clusters;
    p.stages = best.L.stages;
    p.off_ws = best.L.off_ws;
    p.off_a = best.L.off_a;
    p.a_rs = static_cast<uint32_t>(best.nbc) * 64 + 64;
    p.off_asc = best.L.off_asc;
    p.off_red = best.L.off_red;
    p.off_bar = best.L.off_bar;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(best.ks * best.clusters));
    cfg.blockDim = dim3(CF::kThreads);
    cfg.dynamicSmemBytes = best.L.bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(best.ks);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps[0], maps[1], maps[2], maps[3], p);
}

}  // namespace

cudaError_t launch_qdot_mmt(const QdotArgs& a, cudaStream_t stream) {
    if (g_small_kernel != 1 || a.S != nullptr) return cudaErrorNotSupported;
    // (tiny planes, K < 128 or N < 32, are left to the register-fed kernel)
    if (a.M < 1 || a.M > 64 || a.N < kBoxRows || a.K < 128 || a.K % 32 != 0) return cudaErrorNotSupported;
    if (a.K > 0x7fffffffLL || a.N > 0x7fffffffLL - kPassRows) return cudaErrorNotSupported;
    const int64_t KB = a.K / 32;
    // TMA: 16-byte aligned bases, row strides a multiple of 16 bytes
    if ((reinterpret_cast<uintptr_t>(a.W) & 15u) != 0 || (reinterpret_cast<uintptr_t>(a.WS) & 15u) != 0)
        return cudaErrorNotSupported;
    if (a.ws_layout == 0 ? (KB % 4 != 0) : (a.N % 4 != 0)) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(a.A) & 3u) != 0) return cudaErrorNotSupported;

    // weights and scales in boxes of a whole pass (128 rows) and of 32 rows
    CUtensorMap maps[4];
    for (int h = 0; h < 2; ++h) {
        const int rows = h == 0 ? kPassRows : kBoxRows;
        if (!make_map(&maps[2 * h], CU_TENSOR_MAP_DATA_TYPE_UINT8, a.W, a.K, a.N, 1, 128, rows,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorNotSupported;
        const bool ok = a.ws_layout == 0
                            ? make_map(&maps[2 * h + 1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.WS, KB, a.N, 4,
                                       kStageBlocks, rows, CU_TENSOR_MAP_SWIZZLE_NONE)
                            : make_map(&maps[2 * h + 1], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.WS, a.N, KB, 4, rows,
                                       kStageBlocks, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!ok) return cudaErrorNotSupported;
    }

    MmtParams p{};
    p.A = a.A;
    p.AS = a.AS;
    p.C = a.C;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.KB = static_cast<int>(KB);
    p.ntiles = static_cast<int>((a.N + 7) / 8);
    p.ws_layout = a.ws_layout;
    p.vec2 = (reinterpret_cast<uintptr_t>(a.C) & 7u) == 0 && a.N % 2 == 0;
    p.inject_skip = g_skip_stage;
    p.early_weights = a.early_weights;
    p.timeout_cycles = g_timeout;
    const int MT = static_cast<int>((a.M + 15) / 16);
    if (MT == 1) return launch_mt<1>(maps, p, stream);
    if (MT == 2) return launch_mt<2>(maps, p, stream);
    return launch_mt<4>(maps, p, stream);
}

cudaError_t read_and_clear_status_mmt(unsigned* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_pq_status_mmt, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_pq_status_mmt, &zero, sizeof(unsigned));
}

void set_mmt_test_hooks(int inject_skip_stage, unsigned long long timeout_cycles) {
    g_skip_stage = inject_skip_stage;
    g_timeout = timeout_cycles ? timeout_cycles : 4000000000ull;
}

void set_small_kernel(int which) { g_small_kernel = which; }
void set_small_split(int ks) { g_force_ks = ks; }
void small_kernel_config(int* out) {
    for (int i = 0; i < 4; ++i) out[i] = g_last_cfg[i].load(std::memory_order_relaxed);
}
int small_kernel() { return g_small_kernel; }

}  // namespace pq
