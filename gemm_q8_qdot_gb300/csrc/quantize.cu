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

__device__ __forceinline__ uint32_t q_byte(float v, float d) {
    if (d == 0.0f) return 0u;
    int r = __float2int_rn(__fdiv_rn(v, d));  // IEEE x/d, round to nearest even
    r = max(-127, min(127, r));
    return static_cast<uint32_t>(r) & 0xffu;
}

__device__ __forceinline__ uint32_t pack4(float a, float b, float c, float e, float d) {
    return q_byte(a, d) | (q_byte(b, d) << 8) | (q_byte(c, d) << 16) | (q_byte(e, d) << 24);
}

// x may be written by the preceding kernel: coherent load, kept after pdl_wait.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    float4 r;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p) : "memory");
    return r;
}

__global__ void __launch_bounds__(kThreads)
quantize_q8_0_kernel(const float* __restrict__ x, int8_t* __restrict__ q, float* __restrict__ s,
                     int64_t nblocks) {
    // Let the next kernel (typically qdot_t) be scheduled now, so that it can
    // stream its weights while this one runs; then wait for whatever wrote x
    // (and read q, s) before us.
    pdl_trigger();
    pdl_wait();
    const int64_t g = static_cast<int64_t>(blockIdx.x) * kBlocksPerCta + (threadIdx.x >> 2);
    const int sub = threadIdx.x & 3;
    const bool live = g < nblocks;
    float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
    if (live) {
        const float* p = x + g * 32 + sub * 8;
        v0 = ld_stream_f4(p);
        v1 = ld_stream_f4(p + 4);
    }
    float amax = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                       fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
    // every lane of the warp takes part, so the full mask is exact
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    if (live) {
        uint2 packed;
        packed.x = pack4(v0.x, v0.y, v0.z, v0.w, d);
        packed.y = pack4(v1.x, v1.y, v1.z, v1.w, d);
        *reinterpret_cast<uint2*>(q + g * 32 + sub * 8) = packed;
        if (sub == 0) s[g] = d;
    }
}

}  // namespace

cudaError_t launch_quantize(const float* x, int8_t* q, float* s, int64_t rows, int64_t K,
                            cudaStream_t stream) {
    const int64_t nblocks = rows * (K / 32);
    const int64_t grid = (nblocks + kBlocksPerCta - 1) / kBlocksPerCta;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    return launch_pdl(quantize_q8_0_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, stream,
                      x, q, s, nblocks);
}

}  // namespace pq
