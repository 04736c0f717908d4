// Device helpers shared by the kernels of libpq (sm_103a): vector loads with
// cache hints, packed byte arithmetic.  Inline PTX is written here by hand.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace pq {

struct u32x8 {
    uint32_t v[8];
};

// Every global load here is volatile and coherent (no .nc): the kernels are
// launched as programmatic dependents, so data written by the preceding kernel
// is read only after griddepcontrol.wait, and no load may move above it.

// One Q8_0 block of bytes (32 B) in one 256-bit load, not kept in L1: the
// weight stream is touched once per launch.
__device__ __forceinline__ u32x8 ld_stream_v8(const void* p) {
    u32x8 r;
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]),
                   "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
    return r;
}

// Same block, kept in L1: activation rows are re-read by every warp of a CTA.
__device__ __forceinline__ u32x8 ld_cached_v8(const void* p) {
    u32x8 r;
    asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]),
                   "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(p));
    return r;
}

// A 32-byte block from a base that is only 16-byte aligned: two 128-bit loads.
__device__ __forceinline__ u32x8 ld_stream_2v4(const void* p) {
    u32x8 r;
    asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]) : "l"(p));
    asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(static_cast<const char*>(p) + 16));
    return r;
}

// 16-byte-aligned variant of ld_cached_v8.
__device__ __forceinline__ u32x8 ld_cached_2v4(const void* p) {
    u32x8 r;
    asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]) : "l"(p));
    asm volatile("ld.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                 : "l"(static_cast<const char*>(p) + 16));
    return r;
}

// L2 eviction policy of a weight stream.  A launch that reads each weight byte
// once can mark those lines evict_first, so that the stream (many times larger
// than L2 across a model's layers) does not push the small, hot activation rows
// out of L2.  Measured on GB300 (graphs of back-to-back steps, rotating weight
// copies): the fused decode step at K = 4096, N = 4096 goes from 5.2 to 4.8 us
// with it, the Q5_0 decode kernel from 3.91 to 3.82 us; the dp4a qdot_t kernel
// with pre-quantized activations gets slower (4.23 to 4.62 us at M = 1, 31.8 to
// 33.6 us at M = 16), so it does not use it.  A launch whose CTAs read the same
// weights again (several row groups) keeps the normal priority.
__device__ __forceinline__ uint64_t l2_weight_policy(bool read_once) {
    uint64_t pol;
    if (read_once) asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    else asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// A weight block (32 B) with an L2 policy, not kept in L1.
template <bool kV8>
__device__ __forceinline__ u32x8 ld_wblock(const void* p, uint64_t pol) {
    u32x8 r;
    if constexpr (kV8) {
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
                     : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]),
                       "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                     : "l"(p), "l"(pol));
    } else {
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(r.v[0]), "=r"(r.v[1]), "=r"(r.v[2]), "=r"(r.v[3]) : "l"(p), "l"(pol));
        asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.b32 {%0,%1,%2,%3}, [%4], %5;"
                     : "=r"(r.v[4]), "=r"(r.v[5]), "=r"(r.v[6]), "=r"(r.v[7])
                     : "l"(static_cast<const char*>(p) + 16), "l"(pol));
    }
    return r;
}

// A weight scale with an L2 policy.
__device__ __forceinline__ float ld_wscale(const float* p, uint64_t pol) {
    float r;
    asm volatile("ld.global.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(r) : "l"(p), "l"(pol));
    return r;
}

// A 32-bit word of a weight block with an L2 policy (kept in L1: the Q5_0
// kernel reads a 20-byte block as five words, the first brings the line in).
__device__ __forceinline__ uint32_t ld_wword(const void* p, uint64_t pol) {
    uint32_t r;
    asm volatile("ld.global.L2::cache_hint.b32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
    return r;
}

template <bool kV8, bool kStream>
__device__ __forceinline__ u32x8 ld_block(const void* p) {
    if constexpr (kV8) {
        if constexpr (kStream) return ld_stream_v8(p);
        else return ld_cached_v8(p);
    } else {
        if constexpr (kStream) return ld_stream_2v4(p);
        else return ld_cached_2v4(p);
    }
}

__device__ __forceinline__ float ld_f32(const float* p) {
    float r;
    asm volatile("ld.global.f32 %0, [%1];" : "=f"(r) : "l"(p));
    return r;
}

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).  A
// hint only: L2 is the point of coherence, so a later load after pdl_wait still
// sees every write of the preceding kernel.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch.  pdl_trigger lets the next kernel on the
// stream be scheduled now (it still waits for this grid's completion before
// touching our outputs); pdl_wait blocks until the preceding grid has
// completed and its writes are visible.  Both are no-ops for a launch without
// the programmatic-serialization attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// int8x4 -> two f16x2 (exact): bias the bytes to unsigned, put them under the
// f16 exponent of 1024 (0x64xx = 1024 + u), subtract 1152 = 1024 + 128.  lo
// holds bytes 0 and 1 (byte 0 in the low half), hi bytes 2 and 3.
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

// Packed f32 pairs (low word first) and the sm_100+ paired multiply / FMA,
// each element rounded as its scalar counterpart: one instruction for two.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Sum of the 32 signed-byte products of two Q8_0 blocks: eight dp4a.
__device__ __forceinline__ int block_dot(const u32x8& a, const u32x8& w) {
    int s = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) s = __dp4a(static_cast<int>(a.v[t]), static_cast<int>(w.v[t]), s);
    return s;
}

// ---------------------------------------------------------------- Q8_0 quantizer
// Per block of 32: amax = max |x|, d = amax / 127 (IEEE division), q =
// round(x / d) with ties to even, clamped to [-127, 127]; d == 0 gives q = 0.
//
// round(fl(x / d)) without a division per element.  With r = fl(1 / d) (one
// correctly rounded reciprocal per block) and y = fl(x * r), both roundings
// are relative errors of at most 2^-24, and fl(x / d) is one more, so
//   |y - fl(x / d)| <= |x / d| * 3 * 2^-24 <= 1.5 * 2^-16   (|x / d| <= 128,
// which holds for every element of the block since d = fl(amax / 127)).
// Hence if y is more than 2^-14 away from a half-integer, the nearest integer
// to y is the nearest integer to fl(x / d), with no tie to break.  Otherwise
// (a near-tie, about one element in 10^4 for continuous data, or an r that
// is not finite because d is subnormal) the quotient is formed with the IEEE
// division itself.  The result is bit-identical to round(__fdiv_rn(x, d)).
__device__ __forceinline__ int q8_round(float v, float d, float r) {
    const float y = v * r;
    const float n = rintf(y);
    if (fabsf(y - n) < 0.5f - 6.103515625e-05f) return static_cast<int>(n);  // 0.5 - 2^-14
    return __float2int_rn(__fdiv_rn(v, d));
}

__device__ __forceinline__ uint32_t q8_byte(float v, float d, float r) {
    if (d == 0.0f) return 0u;
    const int q = max(-127, min(127, q8_round(v, d, r)));
    return static_cast<uint32_t>(q) & 0xffu;
}

// The block's scale when LANES consecutive lanes share a block: an xor
// butterfly of max over them.  Every lane of the warp must call it
// (full-mask shuffles).
template <int LANES>
__device__ __forceinline__ float q8_scale_of(float amax) {
#pragma unroll
    for (int m = 1; m < LANES; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    return __fdiv_rn(amax, 127.0f);
}

__device__ __forceinline__ float amax4(const float4& v) {
    return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// Four quantized bytes, little-endian in one word.
__device__ __forceinline__ uint32_t q8_pack4(const float4& v, float d, float r) {
    return q8_byte(v.x, d, r) | (q8_byte(v.y, d, r) << 8) | (q8_byte(v.z, d, r) << 16) | (q8_byte(v.w, d, r) << 24);
}

// Four lanes per block, 8 floats each: the block's scale ...
__device__ __forceinline__ float q8_block_scale(const float4& v0, const float4& v1) {
    return q8_scale_of<4>(fmaxf(amax4(v0), amax4(v1)));
}

// ... and this lane's 8 quantized bytes in two words.
__device__ __forceinline__ uint2 q8_pack8(const float4& v0, const float4& v1, float d) {
    const float r = __frcp_rn(d);
    return make_uint2(q8_pack4(v0, d, r), q8_pack4(v1, d, r));
}

// x may be written by the preceding kernel: coherent, kept after pdl_wait.
__device__ __forceinline__ float4 ld_stream_f4(const float* p) {
    float4 r;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p) : "memory");
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

}  // namespace pq
