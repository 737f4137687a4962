// Device helpers shared by the tcgen05 MMQ kernels: UMMA instruction and shared-memory
// descriptors, exact int8 / 4-bit code -> fp16 conversions, and bounded mbarrier waits
// that record a timeout in the calling kernel's error word instead of hanging.
#pragma once

#include <string.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mmq {
namespace umma {

constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // bound on any one wait

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of 8 rows x 16 B
// (8 fp16 along K) stored as 128 contiguous bytes; the next core matrix along K is
// 128 B further (leading-dimension offset), the next 8-row group `sbo` bytes further
// (512 for a K = 32 tile, 256 for a K = 16 tile).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
           (1ull << 46);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) {
    uint32_t o;
    memcpy(&o, &h, 4);
    return o;
}
__device__ __forceinline__ __half2 bits_h2(uint32_t v) {
    __half2 h;
    memcpy(&h, &v, 4);
    return h;
}

// Four signed int8 codes -> four exact fp16 values.  (x + 128) is placed in the low
// mantissa byte of 1024.0 (bits 0x64xx), then 1152 = 1024 + 128 is subtracted.
__device__ __forceinline__ uint2 i8x4_to_f16x4(uint32_t w) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = bits_h2(0x64806480u);
    return make_uint2(h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4140)), bias)),
                      h2_bits(__hsub2(bits_h2(__byte_perm(u, 0x64646464u, 0x4342)), bias)));
}

// Four codes q in 0..15 (one per byte) -> four exact fp16 values sc*q, from the bits of
// 1024 + q and one fused (1024 + q)*sc - 1024*sc (exact: sc*q <= 945).
__device__ __forceinline__ uint2 u4x4_scaled_f16x4(uint32_t w, __half2 sc2, __half2 nsc1024) {
    return make_uint2(h2_bits(__hfma2(bits_h2(__byte_perm(w, 0x64646464u, 0x4140)), sc2, nsc1024)),
                      h2_bits(__hfma2(bits_h2(__byte_perm(w, 0x64646464u, 0x4342)), sc2, nsc1024)));
}

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or the wall
// time limit ran out (then the error word and the abort flag are set).  The abort flag
// and the clock are checked every 64 polls only: a poll is one instruction.  Inlined: a
// call here costs the waiting warp more than the wait itself.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort, unsigned* err) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                atomicOr(err, ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// As wait_bar, with a run-time bound (a device variable the caller has read): for one
// slow-path wait only, so that the hot waits keep their compile-time bound.  A bound of 0
// (a test setting) gives up at once if the phase is not already complete.
__device__ __forceinline__ bool wait_bar_bounded(uint32_t bar, uint32_t parity, volatile int* abort, unsigned* err,
                                                 uint64_t limit_ns) {
    if (limit_ns == 0 && !ptx::mbar_test_wait(bar, parity)) {
        atomicOr(err, ERR_TIMEOUT);
        *abort = 1;
        return false;
    }
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (ptx::globaltimer_ns() - t0 > limit_ns) {
                atomicOr(err, ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// Teardown wait: bounded by time only (used to drain in-flight copies and MMAs).
static __device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity, unsigned* err) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(err, ERR_TIMEOUT);
            return;
        }
    }
}

// Warp-wide wait: every lane polls the same barrier (one broadcast shared-memory read
// per poll) instead of one lane polling in a divergent branch; the vote keeps the
// warp's answer uniform if the wait gave up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned* err) {
    const bool ok = wait_bar(bar, parity, abort, err);
    return __all_sync(0xffffffffu, ok);
}

// Offset of (row r, k-group kg of 8 fp16) in a K-major no-swizzle tile with 8-row-group
// stride sbo.
__device__ __forceinline__ int core_off(int r, int kg, int sbo) { return (r >> 3) * sbo + kg * 128 + (r & 7) * 16; }

// Epilogue of one 128 x 128 output tile, run by 16 warps.  Warp (q = its TMEM lane
// quarter, warp % 4; cg = column group 0..3) owns rows 32q..32q+31 and columns
// 32cg..32cg+31; thread l of the warp owns row 32q + l (TMEM lane) and those 32
// columns.  Item it sits in TMEM slot t = it % DS: D at column t*2*BN, S at
// t*2*BN + BN, read with 32x32b loads of 16 columns, so D and S arrive in the same
// layout and the rescale is an elementwise FMA.  WIDE: all four loads of an item (D
// and S, two 16-column halves: 64 registers) are issued before one wait; otherwise one
// half at a time (32 registers, two waits).  bar_full / bar_empty: the slots' barriers
// (8 bytes apart); each warp arrives once on bar_empty per item.  DOTS: D of item it (=
// block it) is written to dots[m][n][it] instead.  row_map (optional): the tile's row m
// (m < M) is stored to output row row_map[m].
template <bool DOTS, int DS, int BN, bool WIDE>
__device__ __forceinline__ void epilogue_128x128(int q, int cg, int lane, uint32_t tmem, int nitems, uint32_t bar_full,
                                                 uint32_t bar_empty, volatile int* abort, unsigned* err, int M, int N,
                                                 int m0, int n0, int nb, float* __restrict__ out,
                                                 int32_t* __restrict__ dots, const int* __restrict__ row_map = nullptr) {
    const int c0 = cg * 32;
    const int mrow = m0 + 32 * q + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
    unsigned long long acc[16];  // column pairs (c0 + 2i, c0 + 2i + 1)
#pragma unroll
    for (int c = 0; c < 16; ++c) acc[c] = 0ull;
    for (int it = 0; it < nitems; ++it) {
        const int t = it % DS;
        if (!warp_wait(bar_full + 8 * t, (it / DS) & 1, abort, err)) break;
        ptx::tc_fence_after();
        const uint32_t taddr = lane_base + (uint32_t)(t * 2 * BN);
        if (DOTS) {
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
                uint32_t dv[16];
                ptx::tmem_ld16(taddr + 16 * h, dv);
                ptx::tmem_ld_wait(dv);
                if (mrow < M) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int n = n0 + c0 + 16 * h + c;
                        if (n < N) dots[((long long)mrow * N + n) * nb + it] = __float2int_rn(__uint_as_float(dv[c]));
                    }
                }
            }
        } else if (WIDE) {
            uint32_t d0[16], d1[16], s0[16], s1[16];
            ptx::tmem_ld16(taddr, d0);
            ptx::tmem_ld16(taddr + 16, d1);
            ptx::tmem_ld16(taddr + BN, s0);
            ptx::tmem_ld16(taddr + BN + 16, s1);
            ptx::tmem_ld_wait(d0);
            ptx::tmem_ld_wait(d1);
            ptx::tmem_ld_wait(s0);
            ptx::tmem_ld_wait(s1);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                acc[c] = ptx::fma_f32x2(ptx::f2_bits(__uint_as_float(s0[2 * c]), __uint_as_float(s0[2 * c + 1])),
                                        ptx::f2_bits(__uint_as_float(d0[2 * c]), __uint_as_float(d0[2 * c + 1])),
                                        acc[c]);
                acc[8 + c] = ptx::fma_f32x2(ptx::f2_bits(__uint_as_float(s1[2 * c]), __uint_as_float(s1[2 * c + 1])),
                                            ptx::f2_bits(__uint_as_float(d1[2 * c]), __uint_as_float(d1[2 * c + 1])),
                                            acc[8 + c]);
            }
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t dv[16], sv[16];
                ptx::tmem_ld16(taddr + 16 * h, dv);
                ptx::tmem_ld16(taddr + BN + 16 * h, sv);
                ptx::tmem_ld_wait(dv);
                ptx::tmem_ld_wait(sv);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    acc[8 * h + c] =
                        ptx::fma_f32x2(ptx::f2_bits(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])),
                                       ptx::f2_bits(__uint_as_float(dv[2 * c]), __uint_as_float(dv[2 * c + 1])),
                                       acc[8 * h + c]);
            }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(bar_empty + 8 * t);
    }
    if (!DOTS && !*abort && mrow < M) {
        float* orow = out + (long long)(row_map ? row_map[mrow] : mrow) * N + n0 + c0;
        const int ncols = N - (n0 + c0);  // columns of this warp's 32 that exist
        if (ncols >= 32 && (N & 3) == 0) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
                reinterpret_cast<ulonglong2*>(orow)[c] = make_ulonglong2(acc[2 * c], acc[2 * c + 1]);
        } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                if (2 * c < ncols) orow[2 * c] = __uint_as_float((uint32_t)acc[c]);
                if (2 * c + 1 < ncols) orow[2 * c + 1] = __uint_as_float((uint32_t)(acc[c] >> 32));
            }
        }
    }
}

}  // namespace umma
}  // namespace mmq
