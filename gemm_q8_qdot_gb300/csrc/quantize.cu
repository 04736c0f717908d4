// Row quantizer f32 -> Q8_0 ("Quantized built-ins and formats", section
// "Q8_0": signed bytes with one f32 scale per block of 32; activations are
// quantized the same way as weights).
//
// Per block: amax = max |x|, d = amax / 127 (IEEE division), q = round(x / d)
// with ties to even (the spec's round(), "Phobos Language Spec" section 9,
// Elementwise table), clamped to [-127, 127]; d == 0 gives q = 0.
//
// Layout of the work: a Q8_0 block is 128 contiguous bytes of x.  Four lanes
// share a block, each loading 8 floats as two 16-byte vectors; the block's
// amax is a width-4 xor butterfly of max (a lane collective over a 4-lane
// piece); each lane stores its 8 bytes as one 8-byte store and lane 0 of the
// piece stores d.  A warp covers 8 blocks = 1 KB of x, fully coalesced.  Rows
// need no special handling: K % 32 == 0, so block g of the flat [rows*K/32]
// sequence is x[32g : 32g+32] and s[g].  HBM-bound: 4 B read and 1.125 B
// written per element.
#include "pq_internal.h"
#include "pq_device.cuh"

namespace pq {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerCta = kThreads / 4;

// LATE: let the next kernel in only after this one has waited for its own
// predecessor, so that once the next kernel runs, every kernel before this one
// has completed (the one-call step's qdot_t then reads the weights before its
// own wait).  Otherwise let it in at once, so that it can prefetch its weights
// into L2 while this one runs.
template <bool LATE>
__global__ void __launch_bounds__(kThreads)
quantize_q8_0_kernel(const float* __restrict__ x, int8_t* __restrict__ q, float* __restrict__ s,
                     int64_t nblocks) {
    // wait for whatever wrote x (and read q, s) before us
    if constexpr (!LATE) pdl_trigger();
    pdl_wait();
    if constexpr (LATE) pdl_trigger();
    const int64_t g = static_cast<int64_t>(blockIdx.x) * kBlocksPerCta + (threadIdx.x >> 2);
    const int sub = threadIdx.x & 3;
    const bool live = g < nblocks;
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    if (live) {
        const float* p = x + g * 32 + sub * 8;
        v0 = ld_stream_f4(p);
        v1 = ld_stream_f4(p + 4);
    }
    const float d = q8_block_scale(v0, v1);  // every lane of the warp takes part
    if (live) {
        *reinterpret_cast<uint2*>(q + g * 32 + sub * 8) = q8_pack8(v0, v1, d);
        if (sub == 0) s[g] = d;
    }
}

}  // namespace

cudaError_t launch_quantize(const float* x, int8_t* q, float* s, int64_t rows, int64_t K,
                            cudaStream_t stream, bool late_trigger) {
    const int64_t nblocks = rows * (K / 32);
    const int64_t grid = (nblocks + kBlocksPerCta - 1) / kBlocksPerCta;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (late_trigger)
        return launch_pdl(quantize_q8_0_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, stream,
                          x, q, s, nblocks);
    return launch_pdl(quantize_q8_0_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, stream,
                      x, q, s, nblocks);
}

}  // namespace pq
