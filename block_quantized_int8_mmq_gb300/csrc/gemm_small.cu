// Warp-level MMQ for few activation rows (the decode-like regime, bound by the weight
// bytes read from HBM: "When Does a Kernel Win Surface?", sec. "A bottleneck taxonomy",
// bandwidth-roofline decode).
//
// One warp owns one weight row n and up to MT activation rows.  Lane l walks the
// 32-value blocks u = l, l+32, ... of the row: it loads the block's weight codes once
// (Q8_0: 32 int8 at a 2-byte alignment, fetched as aligned words and funnel-shifted;
// Q4_K: the 32 nibbles of sub-block j from the 16-byte aligned nibble chunk, masked to
// 0..15), forms the exact int32 block dot with each activation row by dp4a, and applies
// that block's scale right away in f32 -- the per-32-block rescale in registers.  The
// partial sums are reduced across the warp with shuffles at the end.
// Q4_K adds -dmin*m_j*xs per sub-block ("When Does a Kernel Win Surface?", sec. "Kept
// levers: Vulkan", affine identity; the per-(row, chunk) scales d*sc and -dmin*m as in
// "13 . r7-r8 raw-byte MMQ kernel", sec. 3.2).
#include "common.cuh"

namespace mmq {
namespace {

constexpr int SMALL_WARPS = 8;
constexpr int SMALL_MT = 8;

template <int FMT>
__device__ __forceinline__ void load_weight_block(const uint8_t* __restrict__ wq, long long n, int nb, int u,
                                                  uint32_t (&ww)[8], float& wscale, float& wmin) {
    if (FMT == FMT_Q8_0) {
        const uint8_t* wb = wq + ((long long)n * nb + u) * Q8_0_BYTES;
        wscale = f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(wb)));
        wmin = 0.f;
        const uint8_t* c = wb + 2;
        const int sh = (int)(reinterpret_cast<uintptr_t>(c) & 3) * 8;
        const uint32_t* p = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(c) & ~(uintptr_t)3);
        if (sh == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) ww[i] = __ldg(p + i);
        } else {
            // codes start 2 bytes into an aligned word (sh == 16): words 0..7 cover the
            // f16 scale and codes 0..29, a 2-byte load fetches codes 30..31 without
            // reading past the block
            uint32_t t[9];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = __ldg(p + i);
            t[8] = __ldg(reinterpret_cast<const unsigned short*>(c + 30));
#pragma unroll
            for (int i = 0; i < 8; ++i) ww[i] = __funnelshift_r(t[i], t[i + 1], sh);
        }
    } else {
        const int sb = u >> 3, j = u & 7;
        const uint8_t* sbk = wq + ((long long)n * (nb >> 3) + sb) * Q4_K_BYTES;
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(sbk));  // d, dmin, scale bytes 0..11
        int sc, mn;
        q4_k_scale_min(hdr.y, hdr.z, hdr.w, j, sc, mn);
        wscale = f16_bits_to_f32(hdr.x) * (float)sc;          // exact: 11 x 6 bits
        wmin = f16_bits_to_f32(hdr.x >> 16) * (float)mn;      // exact
        const uint4* qp = reinterpret_cast<const uint4*>(sbk + 16 + 32 * (j >> 1));
        const uint4 a = __ldg(qp), b = __ldg(qp + 1);
        const int shift = (j & 1) * 4;
        const uint32_t raw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) ww[i] = (raw[i] >> shift) & 0x0F0F0F0Fu;
    }
}

template <int FMT>
__global__ void __launch_bounds__(SMALL_WARPS * 32)
k_mmq_small(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ wq, int M, int N, int nb,
            float* __restrict__ out, int32_t* __restrict__ dots) {
    const int lane = threadIdx.x & 31;
    const long long n = (long long)blockIdx.x * SMALL_WARPS + (threadIdx.x >> 5);
    const int m0 = blockIdx.y * SMALL_MT;
    if (n >= N) return;  // uniform per warp
    const int mcount = min(SMALL_MT, M - m0);

    float acc[SMALL_MT];
#pragma unroll
    for (int i = 0; i < SMALL_MT; ++i) acc[i] = 0.f;

    for (int u = lane; u < nb; u += 32) {
        uint32_t ww[8];
        float wscale, wmin;
        load_weight_block<FMT>(wq, n, nb, u, ww, wscale, wmin);
#pragma unroll
        for (int mi = 0; mi < SMALL_MT; ++mi) {
            if (mi < mcount) {
                const uint8_t* xb = xq + ((long long)(m0 + mi) * nb + u) * Q8_1_BYTES;
                const uint32_t hd = __ldg(reinterpret_cast<const uint32_t*>(xb));
                const uint32_t* xc = reinterpret_cast<const uint32_t*>(xb + 4);
                int D = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) D = __dp4a((int)__ldg(xc + i), (int)ww[i], D);
                if (dots) dots[((long long)(m0 + mi) * N + n) * nb + u] = D;
                const float xd = f16_bits_to_f32(hd);
                acc[mi] = fmaf(xd * wscale, (float)D, acc[mi]);
                if (FMT == FMT_Q4_K) acc[mi] = fmaf(-wmin, f16_bits_to_f32(hd >> 16), acc[mi]);
            }
        }
    }
#pragma unroll
    for (int mi = 0; mi < SMALL_MT; ++mi) {
        float v = acc[mi];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0 && mi < mcount && out) out[(long long)(m0 + mi) * N + n] = v;
    }
}

}  // namespace

int small_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                 int32_t* dots, cudaStream_t s) {
    const int nb = (int)(K / QK);
    if ((M + SMALL_MT - 1) / SMALL_MT > 65535) {
        report(fmt == FMT_Q8_0 ? "mmq_gemm_q8_0" : "mmq_gemm_q4_k", MMQ_ERR_SHAPE,
               "the warp-level path takes M <= 524280");
        return MMQ_ERR_SHAPE;
    }
    dim3 grid((unsigned)((N + SMALL_WARPS - 1) / SMALL_WARPS), (unsigned)((M + SMALL_MT - 1) / SMALL_MT));
    const uint8_t* x8 = static_cast<const uint8_t*>(xq);
    const uint8_t* w8 = static_cast<const uint8_t*>(wq);
    if (fmt == FMT_Q8_0)
        k_mmq_small<FMT_Q8_0><<<grid, SMALL_WARPS * 32, 0, s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
    else
        k_mmq_small<FMT_Q4_K><<<grid, SMALL_WARPS * 32, 0, s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
    return launch_status(fmt == FMT_Q8_0 ? "mmq_gemm_q8_0 (small-M)" : "mmq_gemm_q4_k (small-M)");
}

}  // namespace mmq
