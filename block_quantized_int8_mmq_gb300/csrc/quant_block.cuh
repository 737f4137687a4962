// One q8_1 block quantized by four consecutive lanes ("13 . r7-r8 raw-byte MMQ kernel",
// sec. 3.2, the quantize pass: block amax, scale, round, clamp, block sum).  Lane `part`
// (lane % 4) holds values 8*part .. 8*part + 7 of the block; every lane of the warp must
// take part (full-mask shuffles).  Bit-exact arithmetic: d = amax / 127 and each x / d are
// IEEE divisions, rounding to the nearest integer ties to even, codes clamped to
// [-127, 127], s = f16(d * S) with one f32 multiply; a block whose d is 0 gets all-zero
// codes, d and s.  amax is exact under any association, so the shuffle order changes
// nothing.
#pragma once

#include "common.cuh"

namespace mmq {

// w0, w1: this lane's 8 codes (little-endian bytes); hdr: f16 d | f16 s << 16 (the same on
// the four lanes).
__device__ __forceinline__ void quantize_q8_1_part(const float (&v)[8], uint32_t& w0, uint32_t& w1, uint32_t& hdr) {
    const unsigned FULL = 0xffffffffu;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    int sum = 0;
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int q = 0;
        if (d != 0.f) {
            q = __float2int_rn(__fdiv_rn(v[i], d));
            q = max(-127, min(127, q));
        }
        sum += q;
        w[i >> 2] |= (uint32_t)(q & 0xff) << (8 * (i & 3));
    }
    sum += __shfl_xor_sync(FULL, sum, 1);
    sum += __shfl_xor_sync(FULL, sum, 2);
    w0 = w[0];
    w1 = w[1];
    const uint32_t dh = __half_as_ushort(__float2half_rn(d));
    const uint32_t sh = __half_as_ushort(__float2half_rn(__fmul_rn(d, (float)sum)));
    hdr = dh | (sh << 16);
}

}  // namespace mmq
