// MMQ for few activation rows: the decode-like regime, bound by the weight bytes read
// from HBM ("When Does a Kernel Win Surface?", sec. "A bottleneck taxonomy",
// bandwidth-roofline decode).  Kernels, chosen by small_launch at the end of the file:
//   k_mmq_dp4a_stream  one row (two for Q5_K and long K, up to four in a few cases, see
//                      small_launch): per-warp weight streams, dp4a;
//   k_mmq_i8_stream,   up to eight rows per pass on the tensor cores through mma.sync (Q8_0
//   k_mmq_kq_stream    on s8, Q4_K and Q5_K on f16), per-warp rings of 2-D tensor copies;
//   k_mmq_q6_stream    Q6_K, two to eight rows per pass on f16 (K % 512 == 0, N % 8 == 0):
//                      the matrix copied as lines of eight rows, a CTA-wide chunk ring;
//   k_mmq_small_mma, k_mmq_small  shapes the streams do not take (K % 256 != 0).
// Each kernel's own comment describes it.
//
// The two fallbacks.  k_mmq_small: one warp owns one weight row n and up to MT activation
// rows.  Lane l walks the 32-value blocks u = l, l+32, ... of the row: it loads the
// block's weight codes once (Q8_0: 32 int8 at a 2-byte alignment, fetched as aligned words
// and funnel-shifted; Q4_K: the 32 nibbles of sub-block j from the 16-byte aligned nibble
// chunk, masked to 0..15), forms the exact int32 block dot with each activation row by
// dp4a, and applies that block's scale right away in f32 -- the per-32-block rescale in
// registers.  The partial sums are reduced across the warp with shuffles at the end.
// Q4_K adds -dmin*m_j*xs per sub-block ("When Does a Kernel Win Surface?", sec. "Kept
// levers: Vulkan", affine identity; the per-(row, chunk) scales d*sc and -dmin*m as in
// "13 . r7-r8 raw-byte MMQ kernel", sec. 3.2).
//
// For K a multiple of 64, k_mmq_small_mma runs on the tensor cores instead: mma.sync
// m16n8k16 with 16 weight rows as the M side and up to 8 tokens as N, codes converted to
// exact fp16 in registers.  Within one 32-value block the order of k does not change the
// dot product, so both operands use the same permutation of k: thread (g = lane/4, q =
// lane%4) takes the 8 consecutive values 8q..8q+7 of the block, i.e. 8 contiguous bytes of
// a row (Q4_K: one 8-byte load gives the low nibbles of sub-block 2c and the high nibbles
// of 2c+1).  The 16 warps of a CTA share one 16-row tile and split K; each warp issues
// every load of a batch of chunks (codes, scale headers, activation codes and scales)
// before any math, so the DRAM latency is paid once per batch; the warps reduce through
// shared memory at the end.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

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

__device__ __forceinline__ uint32_t h2sub(uint32_t a, uint32_t b) {
    __half2 x = *reinterpret_cast<__half2*>(&a), y = *reinterpret_cast<__half2*>(&b);
    __half2 r = __hsub2(x, y);
    return *reinterpret_cast<uint32_t*>(&r);
}
// 4 signed int8 -> 2 x half2 (exact): bias to unsigned, place in 1024.0's mantissa, subtract 1152
__device__ __forceinline__ void s8x4_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = h2sub(__byte_perm(u, 0x64646464u, 0x4140), 0x64806480u);
    hi = h2sub(__byte_perm(u, 0x64646464u, 0x4342), 0x64806480u);
}
// 4 codes 0..15 (one per byte) -> 2 x half2 (exact)
__device__ __forceinline__ void u4x4_h2(uint32_t w, uint32_t& lo, uint32_t& hi) {
    lo = h2sub(__byte_perm(w, 0x64646464u, 0x4140), 0x64006400u);
    hi = h2sub(__byte_perm(w, 0x64646464u, 0x4342), 0x64006400u);
}

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The 8 code bytes of weight row n, 32-block b, at values 8q..8q+7 (two words).
template <int FMT>
__device__ __forceinline__ uint2 load_w8(const uint8_t* __restrict__ wq, long long n, int nb, int b, int q) {
    if (FMT == FMT_Q4_K) {
        // chunk c = (b/2)%4 of super-block b/8 holds sub-blocks 2c (low) and 2c+1 (high)
        const uint8_t* p = wq + ((long long)n * (nb >> 3) + (b >> 3)) * Q4_K_BYTES + 16 + 32 * ((b >> 1) & 3) + 8 * q;
        return __ldg(reinterpret_cast<const uint2*>(p));
    } else {
        const uint8_t* p = wq + ((long long)n * nb + b) * Q8_0_BYTES + 2 + 8 * q;
        const uint32_t* a = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)3);
        const int sh = (int)(reinterpret_cast<uintptr_t>(p) & 3) * 8;  // 0 or 16
        const uint32_t w0 = __ldg(a), w1 = __ldg(a + 1);
        if (sh == 0) return make_uint2(w0, w1);
        const uint32_t w2 = __ldg(reinterpret_cast<const unsigned short*>(p + 6));
        return make_uint2(__funnelshift_r(w0, w1, 16), __funnelshift_r(w1, w2, 16));
    }
}

// Per-row scale of block b: Q8_0 wd; Q4_K d*sc_j and dmin*m_j.
template <int FMT>
__device__ __forceinline__ void load_wscale(const uint8_t* __restrict__ wq, long long n, int nb, int b, float& ws,
                                            float& wm) {
    if (FMT == FMT_Q4_K) {
        const uint4 h = __ldg(reinterpret_cast<const uint4*>(wq + ((long long)n * (nb >> 3) + (b >> 3)) * Q4_K_BYTES));
        int sc, mn;
        q4_k_scale_min(h.y, h.z, h.w, b & 7, sc, mn);
        ws = f16_bits_to_f32(h.x) * (float)sc;
        wm = f16_bits_to_f32(h.x >> 16) * (float)mn;
    } else {
        ws = f16_bits_to_f32(__ldg(reinterpret_cast<const unsigned short*>(wq + ((long long)n * nb + b) * Q8_0_BYTES)));
        wm = 0.f;
    }
}

constexpr int MMA_WARPS = 16;
constexpr int MMA_BATCH = 1;  // 64-value chunks per warp whose loads are all issued before any math

// Everything one chunk (two 32-blocks) needs, loaded up front.
struct ChunkRegs {
    uint2 w[2][2];       // [row g / g+8][block 2c / 2c+1] (Q4_K: [row][0] holds both sub-blocks)
    uint4 wh[2];         // Q4_K super-block header per row; Q8_0: .x = wd of block 2c, .y = of 2c+1
    uint32_t xa[2][2];   // token g codes: [block][word]
    uint32_t xh[2][2];   // tokens t0 / t1 header (d | s << 16): [block][token]
};

template <int FMT>
__device__ __forceinline__ void load_chunk(ChunkRegs& r, const uint8_t* __restrict__ xq, const uint8_t* __restrict__ wq,
                                           long long row0, long long row1, int nb, int c, int q, int tok, int t0,
                                           int t1, int M) {
    const long long rows[2] = {row0, row1};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        r.w[i][0] = load_w8<FMT>(wq, rows[i], nb, 2 * c, q);
        if (FMT == FMT_Q8_0) {
            r.w[i][1] = load_w8<FMT>(wq, rows[i], nb, 2 * c + 1, q);
            const uint8_t* b0 = wq + ((long long)rows[i] * nb + 2 * c) * Q8_0_BYTES;
            r.wh[i].x = __ldg(reinterpret_cast<const unsigned short*>(b0));
            r.wh[i].y = __ldg(reinterpret_cast<const unsigned short*>(b0 + Q8_0_BYTES));
        } else {
            r.wh[i] = __ldg(reinterpret_cast<const uint4*>(wq + ((long long)rows[i] * (nb >> 3) + (c >> 2)) * Q4_K_BYTES));
        }
    }
#pragma unroll
    for (int sb = 0; sb < 2; ++sb) {
        const int b = 2 * c + sb;
        if (tok < M) {
            const uint32_t* xc = reinterpret_cast<const uint32_t*>(xq + ((long long)tok * nb + b) * Q8_1_BYTES + 4 + 8 * q);
            r.xa[sb][0] = __ldg(xc);
            r.xa[sb][1] = __ldg(xc + 1);
        } else {
            r.xa[sb][0] = r.xa[sb][1] = 0u;
        }
        r.xh[sb][0] = t0 < M ? __ldg(reinterpret_cast<const uint32_t*>(xq + ((long long)t0 * nb + b) * Q8_1_BYTES)) : 0u;
        r.xh[sb][1] = t1 < M ? __ldg(reinterpret_cast<const uint32_t*>(xq + ((long long)t1 * nb + b) * Q8_1_BYTES)) : 0u;
    }
}

template <int FMT>
__global__ void __launch_bounds__(MMA_WARPS * 32, 2)
k_mmq_small_mma(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ wq, int M, int N, int nb,
                float* __restrict__ out, int32_t* __restrict__ dots) {
    __shared__ float red[MMA_WARPS][16][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int n0 = blockIdx.x * 16, m0 = blockIdx.y * 8;
    const long long r0 = min(n0 + g, N - 1), r1 = min(n0 + g + 8, N - 1);  // clamped rows (results discarded)
    const int tok = m0 + g;                                                 // B-fragment token
    const int t0 = m0 + 2 * q, t1 = t0 + 1;                                 // D-fragment tokens
    const int nchunk = nb >> 1;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // (row g, t0), (row g, t1), (row g+8, t0), (row g+8, t1)

    for (int cb = warp; cb < nchunk; cb += MMA_WARPS * MMA_BATCH) {
        ChunkRegs R[MMA_BATCH];
#pragma unroll
        for (int u = 0; u < MMA_BATCH; ++u) {
            const int c = cb + u * MMA_WARPS;
            if (c < nchunk) load_chunk<FMT>(R[u], xq, wq, r0, r1, nb, c, q, tok, t0, t1, M);
        }
#pragma unroll
        for (int u = 0; u < MMA_BATCH; ++u) {
            const int c = cb + u * MMA_WARPS;
            if (c >= nchunk) break;
#pragma unroll
            for (int sb = 0; sb < 2; ++sb) {
                const int b = 2 * c + sb;
                uint32_t a_lo[4], a_hi[4];  // A fragments of the two K=16 mmas (values 8q..8q+3, 8q+4..8q+7)
                float ws[2], wm[2];
                if (FMT == FMT_Q4_K) {
                    const int shift = 4 * sb;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        u4x4_h2((R[u].w[i][0].x >> shift) & 0x0F0F0F0Fu, a_lo[i], a_lo[i + 2]);
                        u4x4_h2((R[u].w[i][0].y >> shift) & 0x0F0F0F0Fu, a_hi[i], a_hi[i + 2]);
                        int sc, mn;
                        q4_k_scale_min(R[u].wh[i].y, R[u].wh[i].z, R[u].wh[i].w, b & 7, sc, mn);
                        ws[i] = f16_bits_to_f32(R[u].wh[i].x) * (float)sc;
                        wm[i] = f16_bits_to_f32(R[u].wh[i].x >> 16) * (float)mn;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        s8x4_h2(R[u].w[i][sb].x, a_lo[i], a_lo[i + 2]);
                        s8x4_h2(R[u].w[i][sb].y, a_hi[i], a_hi[i + 2]);
                        ws[i] = f16_bits_to_f32(sb ? R[u].wh[i].y : R[u].wh[i].x);
                        wm[i] = 0.f;
                    }
                }
                uint32_t b_lo0, b_lo1, b_hi0, b_hi1;
                s8x4_h2(R[u].xa[sb][0], b_lo0, b_lo1);
                s8x4_h2(R[u].xa[sb][1], b_hi0, b_hi1);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(d, a_lo, b_lo0, b_lo1);
                mma16816(d, a_hi, b_hi0, b_hi1);
                if (dots) {
                    const int rr[2] = {n0 + g, n0 + g + 8}, tt[2] = {t0, t1};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (rr[e >> 1] < N && tt[e & 1] < M)
                            dots[((long long)tt[e & 1] * N + rr[e >> 1]) * nb + b] = __float2int_rn(d[e]);
                } else {
                    const float xd0 = f16_bits_to_f32(R[u].xh[sb][0]), xs0 = f16_bits_to_f32(R[u].xh[sb][0] >> 16);
                    const float xd1 = f16_bits_to_f32(R[u].xh[sb][1]), xs1 = f16_bits_to_f32(R[u].xh[sb][1] >> 16);
                    acc[0] = fmaf(xd0 * ws[0], d[0], acc[0]);
                    acc[1] = fmaf(xd1 * ws[0], d[1], acc[1]);
                    acc[2] = fmaf(xd0 * ws[1], d[2], acc[2]);
                    acc[3] = fmaf(xd1 * ws[1], d[3], acc[3]);
                    if (FMT == FMT_Q4_K) {
                        acc[0] = fmaf(-wm[0], xs0, acc[0]);
                        acc[1] = fmaf(-wm[0], xs1, acc[1]);
                        acc[2] = fmaf(-wm[1], xs0, acc[2]);
                        acc[3] = fmaf(-wm[1], xs1, acc[3]);
                    }
                }
            }
        }
    }
    if (dots) return;
    red[warp][g][2 * q] = acc[0];
    red[warp][g][2 * q + 1] = acc[1];
    red[warp][g + 8][2 * q] = acc[2];
    red[warp][g + 8][2 * q + 1] = acc[3];
    __syncthreads();
    if (threadIdx.x < 128) {
        const int rr = threadIdx.x >> 3, tt = threadIdx.x & 7;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < MMA_WARPS; ++w) v += red[w][rr][tt];
        if (n0 + rr < N && m0 + tt < M) out[(long long)(m0 + tt) * N + n0 + rr] = v;
    }
}

// ---------------------------------------------------------------- dp4a stream kernel
// k_mmq_dp4a_stream: for MT <= 2 activation rows, where a tensor-core tile would waste
// most of its 8 token columns, every block dot is formed by dp4a on the raw codes (Q4_K
// nibbles masked to bytes, Q8_0 codes as they are).  The kernel is a set of independent
// weight streams, one per warp, sized so that all CTAs are resident at once: warp gw of
// tw owns the rows gw, gw + tw, ..., and walks them in pieces of up to 16 Q4_K
// super-blocks (2304 B) or 64 Q8_0 blocks (2176 B), each one 1-D bulk async copy into
// the warp's own ring of four slots.  With 16 warps per SM that keeps about 64 copies
// (~150 KB) in flight per SM, enough to cover the HBM latency ("When Does a Kernel Win
// Surface?", sec. "A bottleneck taxonomy": the decode regime is bound by the weight
// bytes); more, smaller copies per SM were measured to stream slower.
//
// A lane owns whole 32-blocks, so each block dot is complete in one lane and its scale
// is applied right there (the per-32-block rescale in registers):
//   Q4_K: lanes 2s and 2s + 1 take super-block s of the piece, halves h = 0 / 1, i.e.
//         nibble chunks 2h and 2h + 1 (sub-blocks 4h .. 4h + 3).  The four 6-bit
//         sub-scales and sub-mins of a half are unpacked byte-parallel from the 12 scale
//         bytes (one word each), the nibbles masked to bytes, and each sub-block adds
//         (d*sc_j * xd) * D - (dmin*m_j) * xs.
//   Q8_0: lane l takes blocks 2l and 2l + 1 (68 bytes at a 4-byte aligned offset, read
//         as 17 words; the first block's codes are funnel-shifted by 16 bits).
// The CTA first copies its MT activation rows into shared memory with 16 bytes of
// padding after every 4 blocks (block b at (b / 4) * 144 + (b % 4) * 32), so that the
// 16-byte reads of lanes 4 or 2 blocks apart fall in distinct banks; f32 xd and xs are
// stored beside them.  The warp reduces with shuffles at the end of a row.
__device__ unsigned int g_small_error;

constexpr int DS_WARPS = 8;
// slot bytes: 16 Q4_K super-blocks (2304 B; a Q8_0 piece, 64 * 34 = 2176 B, fits), 16
// Q5_K super-blocks (2816 B), or 16 Q6_K super-blocks (3360 B) with room for the 16-byte
// granules around them (their rows are only 2-byte aligned: see the copy below)
__host__ __device__ constexpr int ds_slot(int fmt) {
    return fmt == FMT_Q6_K ? 16 * Q6_K_BYTES + 32 : fmt == FMT_Q5_K ? 16 * Q5_K_BYTES : 16 * Q4_K_BYTES;
}
constexpr uint64_t DS_WAIT_LIMIT_NS = 2000000000ull;
constexpr uint32_t DS_SLEEP_NS = 2000;    // suspend hint of one barrier poll
__host__ __device__ constexpr int ds_piece_units(int fmt) { return is_superblock(fmt) ? 16 : 64; }
__host__ __device__ constexpr int ds_unit_bytes(int fmt) { return is_superblock(fmt) ? kq_bytes(fmt) : Q8_0_BYTES; }
__host__ __device__ constexpr int ds_ring_bytes(int fmt, int slots) { return DS_WARPS * slots * (ds_slot(fmt) + 8); }
// activation row stride in shared memory: 144 B per 4 blocks (nb % 8 == 0)
__host__ __device__ constexpr int ds_xrow_bytes(int nb) { return nb / 4 * 144; }
__host__ __device__ constexpr int ds_smem_bytes(int fmt, int mt, int slots, int nb) {
    return ds_ring_bytes(fmt, slots) + mt * (ds_xrow_bytes(nb) + 8 * nb);
}
static_assert(64 * Q8_0_BYTES <= ds_slot(FMT_Q8_0) && (64 * Q8_0_BYTES) % 16 == 0 && ds_slot(FMT_Q4_K) % 16 == 0 &&
                  ds_slot(FMT_Q5_K) % 16 == 0 && ds_slot(FMT_Q6_K) % 16 == 0,
              "slots");

// All lanes of the warp poll the slot's barrier (sleeping in the poll); false on every
// lane after the time limit, with the error recorded.
__device__ __forceinline__ bool ds_wait(uint32_t bar, uint32_t parity) {
    bool done = ptx::mbar_try_wait(bar, parity);
    if (!done) {
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!(done = ptx::mbar_try_wait_sleep(bar, parity, DS_SLEEP_NS)))
            if (ptx::globaltimer_ns() - t0 > DS_WAIT_LIMIT_NS) break;
    }
    done = __all_sync(0xffffffffu, done);
    if (!done && (threadIdx.x & 31) == 0) atomicOr(&g_small_error, ERR_TIMEOUT);
    return done;
}

// byte u of a word as an exact f32 (0..255): the byte placed in the low mantissa bits
// of 2^23 (unit 1), then 2^23 subtracted; byte_f32_div16: the same under 2^19 (unit 1/16)
__device__ __forceinline__ float byte_f32(uint32_t w, int u) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440 + u)) - 8388608.f;
}
__device__ __forceinline__ float byte_f32_div16(uint32_t w, int u) {
    return __uint_as_float(__byte_perm(w, 0x49000000u, 0x7440 + u)) - 524288.f;
}
// dp4a with unsigned bytes in a and signed bytes in b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// The expert-grouped form of the stream (GROUPED): CTA row y takes tile y of the grouping
// kernels' list, up to MT rows of one expert in the sorted order: the weights of that
// expert (wstride bytes apart), its activation rows and output rows through perm.
struct DsGroup {
    const int2* tiles;   // (first sorted row, expert), *ntiles of them
    const int* ntiles;
    const int* offsets;  // offsets[e + 1]: the end of expert e's rows in the sorted order
    const int* perm;     // sorted row -> activation and output row
    long long wstride;   // bytes of one expert's N x K weights
    long long wend;      // bytes of all experts' weights
};

// S: slots per warp; 4 CTAs per SM with 2 slots, 2 CTAs per SM with 4 (64 copies in flight per SM)
template <int FMT, int MT, int S, bool GROUPED>
__global__ void __launch_bounds__(DS_WARPS * 32, S == 2 ? 4 : 2)
k_mmq_dp4a_stream(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ wq, int M, int N, int nb,
                  float* __restrict__ out, int32_t* __restrict__ dots, DsGroup grp) {
    constexpr int PU = ds_piece_units(FMT), UB = ds_unit_bytes(FMT), DS_SLOT = ds_slot(FMT);
    extern __shared__ __align__(128) uint8_t ds_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = ds_smem + warp * S * DS_SLOT;  // this warp's slots
    const uint32_t bar0 = ptx::smem_u32(ds_smem + DS_WARPS * S * DS_SLOT) + 8 * warp * S;
    const int xrow = ds_xrow_bytes(nb);
    uint8_t* xcodes = ds_smem + ds_ring_bytes(FMT, S);                         // [MT][nb/4][144]
    float* xdv = reinterpret_cast<float*>(xcodes + MT * xrow);           // [MT][nb]
    float* xsv = xdv + MT * nb;                                          // [MT][nb]
    // Q6_K keeps, in place of the block sums s, the integer code sums of each block's two
    // 16-value halves (int16 pairs) for the centring term
    uint32_t* xhs = reinterpret_cast<uint32_t*>(xsv);
    int m0 = blockIdx.y * MT, ntok = min(MT, M - m0);
    long long woff = 0;  // byte offset of this CTA's weight matrix
    if constexpr (GROUPED) {
        // the tile list is the grouping kernels' output, and the tile names the expert: wait
        // for them before anything (no weight prefetch ahead of the wait)
        ptx::grid_dep_wait();
        if ((int)blockIdx.y >= *grp.ntiles) return;
        const int2 tl = grp.tiles[blockIdx.y];
        m0 = tl.x;
        ntok = min(MT, grp.offsets[tl.y + 1] - tl.x);
        woff = (long long)tl.y * grp.wstride;
    }
    // activation / output row of the pass's token t
    auto xrow_of = [&](int t) -> long long { return GROUPED ? (long long)grp.perm[m0 + t] : (long long)(m0 + t); };
    const int tw = gridDim.x * DS_WARPS, gw = blockIdx.x * DS_WARPS + warp;
    const int units = is_superblock(FMT) ? nb >> 3 : nb;  // super-blocks or blocks per row
    const int ppr = (units + PU - 1) / PU;             // pieces per row
    const long long row_bytes = (long long)units * UB;
    const int nrows = gw < N ? (N - 1 - gw) / tw + 1 : 0;
    const int total = nrows * ppr;  // pieces of this warp

    auto issue = [&](int q) {  // lane 0: the copy of piece q into slot q % S
        const int r = q / ppr, p = q - r * ppr;
        const long long n = gw + (long long)r * tw;
        const int u0 = p * PU, nu = min(PU, units - u0);
        const uint32_t bar = bar0 + 8 * (q % S);
        if (FMT == FMT_Q6_K) {
            // 210-byte super-blocks leave rows 2-byte aligned: copy the 16-byte granules that
            // hold the piece (the consumer starts at the piece's offset in the first one).
            // The buffer's bytes past its last whole granule come by plain loads instead.
            const long long a = woff + n * row_bytes + (long long)u0 * UB;
            const long long end = GROUPED ? grp.wend : (long long)N * row_bytes;
            const long long a0 = a & ~15ll, lim = end & ~15ll;
            long long a1 = (a + (long long)nu * UB + 15) & ~15ll;
            uint8_t* slot = ring + (q % S) * DS_SLOT;
            if (a1 > lim) {
                for (long long o = lim; o < end; o += 2)
                    *reinterpret_cast<uint16_t*>(slot + (o - a0)) = __ldg(reinterpret_cast<const uint16_t*>(wq + o));
                a1 = lim;
            }
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)(a1 - a0));
            ptx::bulk_load(ptx::smem_u32(slot), wq + a0, (uint32_t)(a1 - a0), bar);
            return;
        }
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)(nu * UB));
        ptx::bulk_load(ptx::smem_u32(ring + (q % S) * DS_SLOT), wq + woff + n * row_bytes + (long long)u0 * UB,
                       (uint32_t)(nu * UB), bar);
    };
    int issued = 0;  // pieces whose copies were issued (kept by every lane)
    if (lane == 0) {
        for (int i = 0; i < S; ++i) ptx::mbar_init(bar0 + 8 * i, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    for (; issued < S && issued < total; ++issued)
        if (lane == 0) issue(issued);
    // Launched as a programmatic dependent: the weights (never written by a kernel of this
    // library) start streaming while the previous kernel on the stream drains; the
    // activations may be its output, so they are read, and anything is written, only after
    // it has completed.  The next kernel may be scheduled from here on.
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();
    // stage the activation rows (rows past M as zeros) while the first pieces arrive
    for (int e = threadIdx.x; e < MT * nb; e += DS_WARPS * 32) {
        const int t = e / nb, b = e - t * nb;
        uint32_t h = 0u, c[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (t < ntok) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(xq + (xrow_of(t) * nb + b) * Q8_1_BYTES);
            h = __ldg(src);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = __ldg(src + 1 + i);
        }
        uint4* dst = reinterpret_cast<uint4*>(xcodes + t * xrow + (b >> 2) * 144 + (b & 3) * QK);
        dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
        dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
        xdv[e] = f16_bits_to_f32(h);
        if (FMT == FMT_Q6_K) {
            int s0 = 0, s1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s0 = __dp4a((int)c[i], 0x01010101, s0);
                s1 = __dp4a((int)c[i + 4], 0x01010101, s1);
            }
            xhs[e] = ((uint32_t)s0 & 0xFFFFu) | ((uint32_t)s1 << 16);
        } else {
            xsv[e] = f16_bits_to_f32(h >> 16);
        }
    }
    __syncthreads();

    bool ok = true;
    int q = 0;  // pieces consumed
    for (int r = 0; r < nrows && ok; ++r) {
        const long long n = gw + (long long)r * tw;
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.f;
        for (int p = 0; p < ppr; ++p, ++q) {
            if (!ds_wait(bar0 + 8 * (q % S), (q / S) & 1)) {
                ok = false;
                break;
            }
            const uint8_t* pc = ring + (q % S) * DS_SLOT;
            const int u0 = p * PU, nu = min(PU, units - u0);
            if (FMT == FMT_Q6_K) {
                const int sl = lane >> 1, h = lane & 1;  // super-block of the piece, half
                if (sl < nu) {
                    // the super-block starts at an even byte of the slot: read 4-byte words from
                    // the word boundary below it and funnel-shift by 0 or 16 bits
                    const int bs = (int)((woff + n * row_bytes + (long long)u0 * UB) & 15) + sl * Q6_K_BYTES;
                    const uint32_t* wa = reinterpret_cast<const uint32_t*>(pc + (bs & ~3));
                    const int fs = (bs & 2) * 8;
                    // half h: low-nibble bytes 64h .. 64h + 63, high-part bytes 128 + 32h ..
                    // 128 + 32h + 31, scales 192 + 8h .. 192 + 8h + 7
                    uint32_t ql[16], qh[8], scw[2];
                    {
                        uint32_t prev = wa[16 * h];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint32_t nx = wa[16 * h + i + 1];
                            ql[i] = __funnelshift_r(prev, nx, fs);
                            prev = nx;
                        }
                        prev = wa[32 + 8 * h];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const uint32_t nx = wa[32 + 8 * h + i + 1];
                            qh[i] = __funnelshift_r(prev, nx, fs);
                            prev = nx;
                        }
                        prev = wa[48 + 2 * h];
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const uint32_t nx = wa[48 + 2 * h + i + 1];
                            scw[i] = __funnelshift_r(prev, nx, fs);
                            prev = nx;
                        }
                    }
                    const float d = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(pc + bs + 208));
                    const int b0 = 8 * (u0 + sl) + 4 * h;  // first block of the half in the row
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const uint8_t* xb = xcodes + t * xrow + (b0 >> 2) * 144;  // blocks b0 .. b0 + 3
                        const float4 xd = *reinterpret_cast<const float4*>(xdv + t * nb + b0);
                        const uint4 hs = *reinterpret_cast<const uint4*>(xhs + t * nb + b0);
                        const float xdu[4] = {xd.x, xd.y, xd.z, xd.w};
                        const uint32_t hsu[4] = {hs.x, hs.y, hs.z, hs.w};
                        float sacc = 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {  // block 4h + u: value 128h + 32u + l
                            const uint4 xa = *reinterpret_cast<const uint4*>(xb + u * QK);
                            const uint4 xc = *reinterpret_cast<const uint4*>(xb + u * QK + 16);
                            uint32_t code[8];  // 6-bit codes 0..63, four per word
#pragma unroll
                            for (int k = 0; k < 8; ++k)
                                code[k] = ((ql[8 * (u & 1) + k] >> (4 * (u >> 1))) & 0x0F0F0F0Fu) |
                                          (((qh[k] >> (2 * u)) & 0x03030303u) << 4);
                            int Da = 0, Db = 0;  // the two 16-value groups
                            Da = dp4a_us(code[0], xa.x, Da);
                            Da = dp4a_us(code[1], xa.y, Da);
                            Da = dp4a_us(code[2], xa.z, Da);
                            Da = dp4a_us(code[3], xa.w, Da);
                            Db = dp4a_us(code[4], xc.x, Db);
                            Db = dp4a_us(code[5], xc.y, Db);
                            Db = dp4a_us(code[6], xc.z, Db);
                            Db = dp4a_us(code[7], xc.w, Db);
                            // centring as a bias term: sum (q - 32) u = dp4a(q, u) - 32 sum u
                            Da -= 32 * (int)(int16_t)(hsu[u] & 0xFFFFu);
                            Db -= 32 * ((int)hsu[u] >> 16);
                            const uint32_t sw = scw[u >> 1] >> (16 * (u & 1));
                            const int D = (int)(int8_t)(sw & 0xFFu) * Da + (int)(int8_t)((sw >> 8) & 0xFFu) * Db;
                            if (dots) {
                                if (t < ntok) dots[((long long)(m0 + t) * N + n) * nb + b0 + u] = D;
                            } else {
                                sacc = fmaf(xdu[u], (float)D, sacc);
                            }
                        }
                        acc[t] = fmaf(d, sacc, acc[t]);
                    }
                }
            } else if (is_kquant(FMT)) {
                const int sl = lane >> 1, h = lane & 1;  // super-block of the piece, half
                if (sl < nu) {
                    const uint8_t* sbk = pc + sl * UB;
                    const uint4 hdr = *reinterpret_cast<const uint4*>(sbk);
                    // sub-blocks 4h + u, u = 0..3: 6-bit scale and min, one per byte
                    const uint32_t sc4 = h ? ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u)) : (hdr.y & 0x3F3F3F3Fu);
                    const uint32_t mn4 =
                        h ? (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u)) : (hdr.z & 0x3F3F3F3Fu);
                    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
                    // Q4_K: sc_j as f32, divided by 16 for the high-nibble sub-blocks (their dot
                    // is formed on the nibble in place, i.e. 16x the code); Q5_K codes are built
                    // whole (nibble | fifth bit << 4).  m_j as f32 (all exact)
                    float scf[4], mnf[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        scf[u] = (FMT == FMT_Q4_K && (u & 1)) ? byte_f32_div16(sc4, u) : byte_f32(sc4, u);
                        mnf[u] = byte_f32(mn4, u);
                    }
                    const int b0 = 8 * (u0 + sl) + 4 * h;  // first block (sub-block 4h) in the row
                    // nibble chunks 2h and 2h + 1: bytes 64h .. 64h + 63 of the nibble bytes
                    const uint4* wc = reinterpret_cast<const uint4*>(sbk + kq_qs_off(FMT) + 64 * h);
                    const uint4 w0 = wc[0], w1 = wc[1], w2 = wc[2], w3 = wc[3];
                    const uint32_t wv[2][8] = {{w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w},
                                               {w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w}};
                    uint32_t qhw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // Q5_K: high-bit bytes 0..31
                    if (FMT == FMT_Q5_K) {
                        const uint4 q0 = *reinterpret_cast<const uint4*>(sbk + 16);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(sbk + 32);
                        qhw[0] = q0.x, qhw[1] = q0.y, qhw[2] = q0.z, qhw[3] = q0.w;
                        qhw[4] = q1.x, qhw[5] = q1.y, qhw[6] = q1.z, qhw[7] = q1.w;
                    }
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const uint8_t* xb = xcodes + t * xrow + (b0 >> 2) * 144;  // blocks b0 .. b0 + 3
                        const float4 xd = *reinterpret_cast<const float4*>(xdv + t * nb + b0);
                        const float4 xs = *reinterpret_cast<const float4*>(xsv + t * nb + b0);
                        const float xdu[4] = {xd.x, xd.y, xd.z, xd.w}, xsu[4] = {xs.x, xs.y, xs.z, xs.w};
                        float sacc = 0.f, macc = 0.f;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {  // sub-block 4h + u: chunk u / 2, low (u even) or high nibbles
                            const uint4 xa = *reinterpret_cast<const uint4*>(xb + u * QK);
                            const uint4 xc = *reinterpret_cast<const uint4*>(xb + u * QK + 16);
                            const uint32_t* cw = wv[u >> 1];
                            uint32_t code[8];
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                if (FMT == FMT_Q5_K)
                                    code[k] = ((cw[k] >> (4 * (u & 1))) & 0x0F0F0F0Fu) |
                                              (((qhw[k] >> (4 * h + u)) & 0x01010101u) << 4);
                                else  // the block dot of a high-nibble sub-block comes out 16x
                                    code[k] = cw[k] & ((u & 1) ? 0xF0F0F0F0u : 0x0F0F0F0Fu);
                            }
                            int D = 0;
                            D = dp4a_us(code[0], xa.x, D);
                            D = dp4a_us(code[1], xa.y, D);
                            D = dp4a_us(code[2], xa.z, D);
                            D = dp4a_us(code[3], xa.w, D);
                            D = dp4a_us(code[4], xc.x, D);
                            D = dp4a_us(code[5], xc.y, D);
                            D = dp4a_us(code[6], xc.z, D);
                            D = dp4a_us(code[7], xc.w, D);
                            if (dots) {
                                const bool x16 = FMT == FMT_Q4_K && (u & 1);
                                if (t < ntok) dots[((long long)(m0 + t) * N + n) * nb + b0 + u] = x16 ? D >> 4 : D;
                            } else {
                                sacc = fmaf(scf[u], xdu[u] * (float)D, sacc);
                                macc = fmaf(mnf[u], xsu[u], macc);
                            }
                        }
                        // (d * sc_j * xd) * D - (dmin * m_j) * xs summed over the half's 4 sub-blocks
                        acc[t] = fmaf(d, sacc, acc[t]);
                        acc[t] = fmaf(-dmin, macc, acc[t]);
                    }
                }
            } else if (2 * lane < nu) {
                // blocks 2l and 2l + 1 of the piece: 68 bytes at offset 68l (4-byte aligned) =
                // [wd0 | 32 codes | wd1 | 32 codes]; nu is even (K % 256 == 0)
                const uint32_t* wp = reinterpret_cast<const uint32_t*>(pc + lane * 2 * Q8_0_BYTES);
                uint32_t w[17];
#pragma unroll
                for (int e = 0; e < 17; ++e) w[e] = wp[e];
                const float wd0 = f16_bits_to_f32(w[0]), wd1 = f16_bits_to_f32(w[8] >> 16);
                const int b0 = u0 + 2 * lane;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const uint8_t* xb = xcodes + t * xrow + (b0 >> 2) * 144 + (b0 & 3) * QK;  // blocks b0, b0 + 1
                    const uint4 xa0 = *reinterpret_cast<const uint4*>(xb);
                    const uint4 xa1 = *reinterpret_cast<const uint4*>(xb + 16);
                    const uint4 xb0 = *reinterpret_cast<const uint4*>(xb + 32);
                    const uint4 xb1 = *reinterpret_cast<const uint4*>(xb + 48);
                    int D0 = 0, D1 = 0;
                    D0 = __dp4a((int)__funnelshift_r(w[0], w[1], 16), (int)xa0.x, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[1], w[2], 16), (int)xa0.y, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[2], w[3], 16), (int)xa0.z, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[3], w[4], 16), (int)xa0.w, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[4], w[5], 16), (int)xa1.x, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[5], w[6], 16), (int)xa1.y, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[6], w[7], 16), (int)xa1.z, D0);
                    D0 = __dp4a((int)__funnelshift_r(w[7], w[8], 16), (int)xa1.w, D0);
                    D1 = __dp4a((int)w[9], (int)xb0.x, D1);
                    D1 = __dp4a((int)w[10], (int)xb0.y, D1);
                    D1 = __dp4a((int)w[11], (int)xb0.z, D1);
                    D1 = __dp4a((int)w[12], (int)xb0.w, D1);
                    D1 = __dp4a((int)w[13], (int)xb1.x, D1);
                    D1 = __dp4a((int)w[14], (int)xb1.y, D1);
                    D1 = __dp4a((int)w[15], (int)xb1.z, D1);
                    D1 = __dp4a((int)w[16], (int)xb1.w, D1);
                    if (dots) {
                        if (t < ntok) {
                            dots[((long long)(m0 + t) * N + n) * nb + b0] = D0;
                            dots[((long long)(m0 + t) * N + n) * nb + b0 + 1] = D1;
                        }
                    } else {
                        const float2 xd = *reinterpret_cast<const float2*>(xdv + t * nb + b0);
                        acc[t] = fmaf(wd0 * xd.x, (float)D0, acc[t]);
                        acc[t] = fmaf(wd1 * xd.y, (float)D1, acc[t]);
                    }
                }
            }
            // every lane is done with the slot: refill it with the piece S ahead
            __syncwarp();
            if (issued < total) {
                if (lane == 0) {
                    ptx::fence_proxy_async_smem();
                    issue(issued);
                }
                ++issued;
            }
        }
        if (!ok) break;
        if (!dots) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0 && t < ntok) out[xrow_of(t) * N + n] = v;
            }
        }
    }
    if (!ok && lane == 0) {
        // copies still in flight must land before the CTA exits
        for (int k = q; k < issued; ++k) {
            const uint64_t t0 = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar0 + 8 * (k % S), (k / S) & 1))
                if (ptx::globaltimer_ns() - t0 > DS_WAIT_LIMIT_NS) break;
        }
    }
}

// GROUPED: grid row y takes tile y of the grouping's list (gtiles rows of CTAs, those past
// the list's length return at once)
template <int FMT, int MT, int S, bool GROUPED = false>
int launch_dp4a_stream_s(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                         int32_t* dots, cudaStream_t s, const char* fn, const DsGroup& grp = DsGroup{},
                         int64_t gtiles = 0) {
    const int smem = ds_smem_bytes(FMT, MT, S, nb);
    static SmemAttr attr;
    if (smem > 48 * 1024) {
        const int e = ensure_smem((const void*)k_mmq_dp4a_stream<FMT, MT, S, GROUPED>, smem, attr);
        if (e != MMQ_OK) {
            report(fn, e, "shared-memory request refused");
            return e;
        }
    }
    // every CTA resident at once (as many per SM as the launch bounds and shared memory
    // allow), and the rows dealt out evenly: rows per warp = ceil(N / warps that fit),
    // then only as many CTAs as that needs
    const DeviceShape ds = device_shape();
    const int per_sm = std::max(1, std::min(S == 2 ? 4 : 2, ds.smem_per_sm / (smem + 1024)));
    const int64_t max_warps = (int64_t)ds.sms * per_sm * DS_WARPS;
    // grouped: 16 weight rows per warp (a CTA stages its tile's activations once for 128
    // rows; measured against 4, 8 and 32 on 128 experts of 768 x 2048: the fastest or within
    // 2 % at 1 to 16 rows per expert)
    const int64_t rpw = GROUPED ? 16 : (N + max_warps - 1) / max_warps;
    const int64_t ctas = (N + DS_WARPS * rpw - 1) / (DS_WARPS * rpw);
    dim3 grid((unsigned)ctas, (unsigned)(GROUPED ? gtiles : (M + MT - 1) / MT));
    {
        ProfScope ps("k_mmq_dp4a_stream", s);
        return pdl_status(launch_pdl(k_mmq_dp4a_stream<FMT, MT, S, GROUPED>, grid, dim3(DS_WARPS * 32), (size_t)smem, s,
                                     x8, w8, (int)M, (int)N, nb, out, dots, grp),
                          fn);
    }
}

// the grouped stream for tiles of mt rows (1, 2 or 4), slots as for that many dense rows
template <int FMT>
int launch_dp4a_grouped(const uint8_t* x8, const uint8_t* w8, int64_t R, int64_t N, int nb, int mt, float* out,
                        cudaStream_t s, const char* fn, const DsGroup& g, int64_t gtiles) {
    if (mt <= 1)
        return FMT == FMT_Q6_K
                   ? launch_dp4a_stream_s<FMT, 1, 4, true>(x8, w8, R, N, nb, out, nullptr, s, fn, g, gtiles)
                   : launch_dp4a_stream_s<FMT, 1, 2, true>(x8, w8, R, N, nb, out, nullptr, s, fn, g, gtiles);
    if (mt <= 2) return launch_dp4a_stream_s<FMT, 2, 4, true>(x8, w8, R, N, nb, out, nullptr, s, fn, g, gtiles);
    return launch_dp4a_stream_s<FMT, 4, 4, true>(x8, w8, R, N, nb, out, nullptr, s, fn, g, gtiles);
}

// Two slots and four CTAs per SM (more warps to hide the math) for one activation row;
// four slots and two CTAs per SM for two, and for Q6_K's one row (measured best for each).
template <int FMT>
int launch_dp4a_stream(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                       int32_t* dots, cudaStream_t s, const char* fn) {
    if (M <= 1)  // Q6_K's slower math keeps more pieces in flight per warp
        return FMT == FMT_Q6_K ? launch_dp4a_stream_s<FMT, 1, 4>(x8, w8, M, N, nb, out, dots, s, fn)
                               : launch_dp4a_stream_s<FMT, 1, 2>(x8, w8, M, N, nb, out, dots, s, fn);
    if (M <= 2) return launch_dp4a_stream_s<FMT, 2, 4>(x8, w8, M, N, nb, out, dots, s, fn);
    return launch_dp4a_stream_s<FMT, 4, 4>(x8, w8, M, N, nb, out, dots, s, fn);
}

// ---------------------------------------------------------------- tensor-core streams
// Two kernels for up to 8 activation rows per pass (grid.y = ceil(M/8) passes), both on the
// tensor cores through mma.sync ("When the Product Won't Collapse", sec. "The obstruction":
// one exact integer dot per 32-block; "13 . r7-r8 raw-byte MMQ kernel", sec. 2), 16 weight
// rows x 8 tokens x one whole 32-block at a time, from the raw codes:
//   k_mmq_i8_stream  Q8_0: m16n8k32 s8 x s8 -> s32 on the codes as they are;
//   k_mmq_kq_stream  Q4_K, Q5_K: two m16n8k16 f16 MMAs per block on exact f16 operands
//                    (on this part the s8 form runs at 69 cycles per MMA per SM sub-
//                    partition, the f16 form at 9 per k16 half; both measured).
// Common structure.  A CTA owns `tpc` consecutive weight boxes (16 rows; 32 for the K-quant
// kernel when there are enough); its warps split each box's K round-robin in pieces (warp w
// takes pieces w, w + W, ...), a piece being the box's rows x one super-block or x 8 Q8_0
// blocks, brought by one 2-D tensor copy into the warp's own ring (rows past N arrive as
// zeros).  The piece's activations (the pass's q8_1 rows x its 8 blocks) come by one more
// tensor copy into the warp's activation slots and serve all of the CTA's boxes.  k is
// permuted identically in A and B, which leaves every block dot unchanged.  The block dots
// are rescaled in registers as they come, in packed f32 pairs; the warps' partial sums of
// a box meet in shared memory at the end, in each warp's weight ring (every copy into it
// consumed by then).  Needs K % 256 == 0.
constexpr int IS_WARPS = 8;
constexpr int IS_XROW = 8 * Q8_1_BYTES;  // one activation row's 8 blocks: 288 B
constexpr int IS_ASLOT = 8 * IS_XROW;    // a piece's activations, 8 rows: 2304 B
constexpr int IS_MAX_TPC = 4;
constexpr int IS_MAGIC = 0x4B400000;                                 // bit pattern of 1.5 * 2^23
constexpr unsigned long long IS_NEG_MAGIC2 = 0xCB400000CB400000ull;  // (-1.5 * 2^23, -1.5 * 2^23)

// (a, b) as an exact f32 pair, for |a|, |b| < 2^22: an int32 v added to the bit pattern of
// 1.5 * 2^23 is the float 1.5 * 2^23 + v, and subtracting 1.5 * 2^23 leaves v exactly
// (no integer-to-float converter)
__device__ __forceinline__ unsigned long long is_exact2(int a, int b) {
    return ptx::add_f32x2(ptx::f2_bits(__int_as_float(a + IS_MAGIC), __int_as_float(b + IS_MAGIC)), IS_NEG_MAGIC2);
}
__device__ __forceinline__ unsigned long long is_splat2(float v) { return ptx::f2_bits(v, v); }
// an f16 pair as an f32 pair
__device__ __forceinline__ unsigned long long is_xd2(uint32_t h2) {
    return ptx::f2_bits(f16_bits_to_f32(h2), f16_bits_to_f32(h2 >> 16));
}
// two bytes of w (0..63, picked by sel) as an exact f16 pair: with 0x64 above it a byte b is
// the f16 1024 + b, and 1024 is subtracted
__device__ __forceinline__ uint32_t is_byte_pair_f16(uint32_t w, uint32_t sel) {
    const uint32_t h = __byte_perm(w, 0x64646464u, sel);
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(0x64006400u));
    return d;
}

__device__ __forceinline__ void mma_s8_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}
// 16 x 8 x 8, f16 operands, f32 result from zero: rows g / g + 8 x columns 2q, 2q + 1 in d
__device__ __forceinline__ void mma_f16_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%7, %7, %7, %7};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "f"(0.f));
}

// Per-warp pipeline bookkeeping shared by both kernels: the weight ring's copy schedule
// (piece-major: a piece's activations serve all the CTA's tiles) without divisions.
struct IsSchedule {
    int k, tl;  // piece and tile of the next copy to issue
};

// ------------------------------------------ Q8_0: k_mmq_i8_stream
// Two weight slots and two activation slots per warp.  A thread loads its piece's codes
// (B) and the f16 xd of its two tokens into registers once per piece.  Each dot D (|D| <=
// 32 * 127 * 128 < 2^22) is made an exact f32 as above and accumulated as acc += (d_w * xd)
// * D, one pair per weight row and the thread's two tokens.
constexpr int I8_SLOTS = 2, I8_ASLOTS = 2;
constexpr int I8_SLOT = 16 * 8 * Q8_0_BYTES;  // 4352
constexpr int I8_WARP_BYTES = I8_SLOTS * I8_SLOT + I8_ASLOTS * IS_ASLOT;
constexpr int I8_SMEM = IS_WARPS * (I8_WARP_BYTES + 8 * (I8_SLOTS + I8_ASLOTS));
static_assert(I8_SMEM <= 110 * 1024 && I8_SLOT % 128 == 0 && IS_ASLOT % 128 == 0, "two CTAs per SM");
static_assert(IS_MAX_TPC * 16 * 8 * 4 <= I8_SLOTS * I8_SLOT, "a warp's partial sums fit in its weight ring");

template <bool DOTS, bool SPLIT = false>
__global__ void __launch_bounds__(IS_WARPS * 32, 2)
k_mmq_i8_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmXl, int M, int N,
                int nb, int tpc, float* __restrict__ out, long long pstride, int32_t* __restrict__ dots) {
    constexpr int S = I8_SLOTS, SA = I8_ASLOTS, SLOT = I8_SLOT, RB = 8 * Q8_0_BYTES, WB = I8_WARP_BYTES;
    extern __shared__ __align__(128) uint8_t is_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    uint8_t* ring = is_smem + warp * WB;  // S weight slots, then SA activation slots
    uint8_t* aring = ring + S * SLOT;
    const uint32_t bar0 = ptx::smem_u32(is_smem + IS_WARPS * WB) + 8 * (S + SA) * warp;
    const uint32_t abar0 = bar0 + 8 * S;
    const int ntiles = (N + 15) / 16;
    const int t0 = blockIdx.x * tpc, nt = min(tpc, ntiles - t0);
    // SPLIT (K split over the grid's z): this CTA's groups of 8 blocks are pz0 .. pz0 +
    // npieces - 1, its partial outputs go to slab z of `out` (pstride floats apart)
    int pz0 = 0, npieces = nb / 8;
    if constexpr (SPLIT) {
        pz0 = (int)((long long)blockIdx.z * (nb / 8) / gridDim.z);
        npieces = (int)((long long)(blockIdx.z + 1) * (nb / 8) / gridDim.z) - pz0;
        out += blockIdx.z * pstride;
    }
    const int my = warp < npieces ? (npieces - 1 - warp) / IS_WARPS + 1 : 0;  // this warp's pieces per tile
    const int total = nt * my;
    const int m0 = blockIdx.y * 8;
    const bool h0ok = m0 + 2 * q < M, h1ok = m0 + 2 * q + 1 < M;  // the D fragment's tokens 2q, 2q + 1

    IsSchedule next{0, 0};
    auto issue = [&](int i) {  // lane 0: the copy of this warp's weight piece i into slot i % S
        const uint32_t bar = bar0 + 8 * (i % S);
        ptx::mbar_arrive_expect_tx(bar, SLOT);  // the whole box, zero-filled rows included
        ptx::tma_load_2d(ptx::smem_u32(ring + (i % S) * SLOT), &tmW, bar, (pz0 + warp + next.k * IS_WARPS) * (RB / 8),
                         (t0 + next.tl) * 16);
    };
    auto advance = [&]() {
        if (++next.tl == nt) next.tl = 0, ++next.k;
    };
    // the pass's activation rows: a box of min(8, M - m0) rows (rows past M are not copied;
    // their slot rows only ever reach outputs that are not stored)
    const bool lastp = blockIdx.y == gridDim.y - 1;
    const uint32_t abytes = (uint32_t)min(M - m0, 8) * IS_XROW;
    auto issue_acts = [&](int k) {  // lane 0: the activations of this warp's piece k into slot k % SA
        const uint32_t bar = abar0 + 8 * (k % SA);
        ptx::mbar_arrive_expect_tx(bar, abytes);
        ptx::tma_load_2d(ptx::smem_u32(aring + (k % SA) * IS_ASLOT), lastp ? &tmXl : &tmX, bar,
                         (pz0 + warp + k * IS_WARPS) * (IS_XROW / 8), m0);
    };
    int issued = 0, aissued = 0;
    if (lane == 0) {
        ptx::tma_prefetch_desc(&tmW);
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmXl);
        for (int i = 0; i < S + SA; ++i) ptx::mbar_init(bar0 + 8 * i, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    for (; issued < S && issued < total; ++issued, advance())
        if (lane == 0) issue(issued);
    // programmatic dependent: the weight pieces above are in flight; the activations are
    // read, and results written, only after the previous kernel on the stream has completed
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();
    for (; aissued < SA && aissued < my; ++aissued)
        if (lane == 0) issue_acts(aissued);

    bool ok = true;
    int i = 0, ka = 0;  // weight and activation slots consumed
    unsigned long long acc[IS_MAX_TPC][2];  // per tile: rows g / g + 8, tokens (2q, 2q + 1)
#pragma unroll
    for (int tl = 0; tl < IS_MAX_TPC; ++tl) acc[tl][0] = acc[tl][1] = 0ull;
    for (int k = 0; k < my && ok; ++k) {
        const int b0 = 8 * (pz0 + warp + k * IS_WARPS);  // first block of the piece
        if (!ds_wait(abar0 + 8 * (k % SA), (k / SA) & 1)) {
            ok = false;
            break;
        }
        ++ka;
        // B fragments (codes 8q .. 8q + 7 of token g) and the f16 xd of tokens 2q, 2q + 1
        const uint8_t* as = aring + (k % SA) * IS_ASLOT;
        uint32_t bw[8][2], xh2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t* cb = reinterpret_cast<const uint32_t*>(as + g * IS_XROW + j * Q8_1_BYTES + 4 + 8 * q);
            bw[j][0] = cb[0];
            bw[j][1] = cb[1];
            const uint32_t e0 = *reinterpret_cast<const uint32_t*>(as + 2 * q * IS_XROW + j * Q8_1_BYTES);
            const uint32_t e1 = *reinterpret_cast<const uint32_t*>(as + (2 * q + 1) * IS_XROW + j * Q8_1_BYTES);
            xh2[j] = __byte_perm(e0, e1, 0x5410);
        }
        // every lane holds its copy: the slot takes the piece SA ahead
        __syncwarp();
        if (aissued < my) {
            if (lane == 0) {
                ptx::fence_proxy_async_smem();
                issue_acts(aissued);
            }
            ++aissued;
        }
#pragma unroll
        for (int tl = 0; tl < IS_MAX_TPC; ++tl) {
            if (tl >= nt) break;
            const int n0 = (t0 + tl) * 16;
            if (!ds_wait(bar0 + 8 * (i % S), (i / S) & 1)) {
                ok = false;
                break;
            }
            const uint8_t* sl = ring + (i % S) * SLOT;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // codes 8q .. 8q + 7 of block j of rows g and g + 8: 2-byte aligned, read as
                // aligned words and funnel-shifted (a third word only when the shift is 16)
                const int off = j * Q8_0_BYTES + 2 + 8 * q, sh = (off & 3) * 8;
                const uint32_t* pg = reinterpret_cast<const uint32_t*>(sl + g * RB + (off & ~3));
                const uint32_t* ph = reinterpret_cast<const uint32_t*>(sl + (g + 8) * RB + (off & ~3));
                const uint32_t g0 = pg[0], g1 = pg[1], g2 = sh ? pg[2] : 0u;
                const uint32_t e0 = ph[0], e1 = ph[1], e2 = sh ? ph[2] : 0u;
                int D[4];
                mma_s8_16832(D, __funnelshift_r(g0, g1, sh), __funnelshift_r(e0, e1, sh), __funnelshift_r(g1, g2, sh),
                             __funnelshift_r(e1, e2, sh), bw[j][0], bw[j][1]);
                if constexpr (DOTS) {
                    const int b = b0 + j;
                    if (h0ok && n0 + g < N) dots[((long long)(m0 + 2 * q) * N + n0 + g) * nb + b] = D[0];
                    if (h1ok && n0 + g < N) dots[((long long)(m0 + 2 * q + 1) * N + n0 + g) * nb + b] = D[1];
                    if (h0ok && n0 + g + 8 < N) dots[((long long)(m0 + 2 * q) * N + n0 + g + 8) * nb + b] = D[2];
                    if (h1ok && n0 + g + 8 < N) dots[((long long)(m0 + 2 * q + 1) * N + n0 + g + 8) * nb + b] = D[3];
                    continue;
                }
                const float wg = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sl + g * RB + j * Q8_0_BYTES));
                const float wh =
                    f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(sl + (g + 8) * RB + j * Q8_0_BYTES));
                const unsigned long long xd = is_xd2(xh2[j]);
                acc[tl][0] = ptx::fma_f32x2(is_exact2(D[0], D[1]), ptx::mul_f32x2(is_splat2(wg), xd), acc[tl][0]);
                acc[tl][1] = ptx::fma_f32x2(is_exact2(D[2], D[3]), ptx::mul_f32x2(is_splat2(wh), xd), acc[tl][1]);
            }
            // every lane is done with the slot: refill it with the piece S ahead
            __syncwarp();
            if (issued < total) {
                if (lane == 0) {
                    ptx::fence_proxy_async_smem();
                    issue(issued);
                }
                ++issued;
                advance();
            }
            ++i;
        }
    }
    if (!ok && lane == 0) {
        // copies still in flight must land before the CTA exits
        for (int k2 = i; k2 < issued; ++k2) {
            const uint64_t tb = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar0 + 8 * (k2 % S), (k2 / S) & 1))
                if (ptx::globaltimer_ns() - tb > DS_WAIT_LIMIT_NS) break;
        }
        for (int k2 = ka; k2 < aissued; ++k2) {
            const uint64_t tb = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(abar0 + 8 * (k2 % SA), (k2 / SA) & 1))
                if (ptx::globaltimer_ns() - tb > DS_WAIT_LIMIT_NS) break;
        }
    }
    if (DOTS) return;
    if (ok && my > 0) {
        // this warp's partial sums, [tile][row][token], over its weight ring
        float* rw = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int tl = 0; tl < IS_MAX_TPC; ++tl) {
            if (tl >= nt) break;
            *reinterpret_cast<unsigned long long*>(rw + (tl * 16 + g) * 8 + 2 * q) = acc[tl][0];
            *reinterpret_cast<unsigned long long*>(rw + (tl * 16 + g + 8) * 8 + 2 * q) = acc[tl][1];
        }
    }
    if (__syncthreads_or(!ok)) return;
    const int nw = min(npieces, IS_WARPS);  // warps that hold partial sums
    for (int e = threadIdx.x; e < nt * 16 * 8; e += IS_WARPS * 32) {
        const int tl = e >> 7, r = (e >> 3) & 15, tok = e & 7;
        float v = 0.f;
        for (int w = 0; w < nw; ++w) v += reinterpret_cast<const float*>(is_smem + w * WB)[e];
        const int n = (t0 + tl) * 16 + r;
        if (n < N && m0 + tok < M) out[(long long)(m0 + tok) * N + n] = v;
    }
}

// ------------------------------------------ Q4_K, Q5_K: k_mmq_kq_stream
// Each 32-block dot is two f16 MMAs (m16n8k16, f32 accumulation) on exact operands.  The
// weight codes need no conversion: a code c <= 1023 in the low bits of an f16 half is the
// subnormal c * 2^-24.  Masking a word of packed nibbles with 0x000F000F leaves two codes
// of a sub-block j (j even) as an f16 pair; the high nibbles of the same bytes (j odd),
// masked in place with 0x00F000F0, are 16 c * 2^-24, and the factor 16 goes into the
// sub-scale (sc_j / 16); the other two bytes of the word take one shift.  Q5_K adds its
// fifth bit in place (16 * 2^-24, or 256 * 2^-24 above a high nibble).  The int8
// activation codes are f16 integers, formed once per piece (byte + 128 under the f16
// 1024 bias, 1152 subtracted).  Every product is an integer times 2^-24 (2^-20 with the
// factor 16), every partial sum below 2^24 units: the two MMAs give the block dot exactly
// (measured exact on this part, subnormal operands included).  The k order inside a
// block is permuted identically on both sides: thread (g, q) owns values 8q .. 8q + 7 of
// the block, k slots (2q, 2q + 1) of the first MMA taking values (8q, 8q + 2), slots
// (2q + 8, 2q + 9) values (8q + 1, 8q + 3), and the second MMA the same four higher.
// Rescale, in packed f32 pairs over the thread's two tokens: S_row += (sc_j, sc_j) * (xd,
// xd') * (D, D') per block, then per super-block acc += d * 2^24 * S - dmin * (sum_j m_j *
// xs_j), the min term one m16n8k8 f16 MMA per tile (6-bit m_j and f16 xs_j are exact f16
// operands, products exact, f32 accumulation).
// A piece's activation codes and xd stay in registers for all of the CTA's tiles; the raw
// q8_1 rows come by tensor copy into two slots per warp (the next piece's while this one
// computes).  A weight copy brings BOXR = 32 rows (two tiles) x one super-block when there
// are enough 32-row boxes to fill the GPU, else 16 rows: the copy engine streams 4.6 KB
// boxes near the HBM rate and 2.3 KB boxes well below it (measured, 16 warps per SM,
// nothing consuming).
__host__ __device__ constexpr int ks_warps(int fmt, int boxr) { return boxr == 16 ? 8 : (fmt == FMT_Q4_K ? 8 : 7); }
__host__ __device__ constexpr int ks_slots(int fmt, int boxr) { return boxr == 16 ? 3 : 2; }
__host__ __device__ constexpr int ks_slot(int fmt, int boxr) { return boxr * kq_bytes(fmt); }
__host__ __device__ constexpr int ks_max_boxes(int boxr) { return boxr == 16 ? 4 : 2; }  // per CTA
constexpr int KS_ASLOTS = 2;
__host__ __device__ constexpr int ks_warp_bytes(int fmt, int boxr) {
    return ks_slots(fmt, boxr) * ks_slot(fmt, boxr) + KS_ASLOTS * IS_ASLOT;
}
__host__ __device__ constexpr int ks_smem_bytes(int fmt, int boxr) {
    return ks_warps(fmt, boxr) * (ks_warp_bytes(fmt, boxr) + 8 * (ks_slots(fmt, boxr) + KS_ASLOTS));
}
constexpr int KS_SMEM_MAX = 113 * 1024;  // two CTAs per SM
static_assert(ks_smem_bytes(FMT_Q4_K, 16) <= KS_SMEM_MAX && ks_smem_bytes(FMT_Q5_K, 16) <= KS_SMEM_MAX &&
                  ks_smem_bytes(FMT_Q4_K, 32) <= KS_SMEM_MAX && ks_smem_bytes(FMT_Q5_K, 32) <= KS_SMEM_MAX,
              "two CTAs per SM");
static_assert(ks_slot(FMT_Q4_K, 16) % 128 == 0 && ks_slot(FMT_Q5_K, 16) % 128 == 0, "128-byte aligned slots");
static_assert(4 * 16 * 8 * 4 <= 2 * ks_slot(FMT_Q4_K, 16), "a warp's partial sums fit in its weight ring");

// 16 x 8 x 16, f16 operands, f32 accumulation: from zero, and in place
__device__ __forceinline__ void mma_f16_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// bytes (sel) of four int8 codes (u = codes ^ 0x80808080, i.e. code + 128) as an exact f16 pair
__device__ __forceinline__ uint32_t ks_code_pair(uint32_t u, uint32_t sel) {
    uint32_t h = __byte_perm(u, 0x64646464u, sel), d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(h), "r"(0xE480E480u));  // - 1152
    return d;
}

template <int FMT, int BOXR, bool DOTS, bool SPLIT = false>
__global__ void __launch_bounds__(ks_warps(FMT, BOXR) * 32, 2)
k_mmq_kq_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmXl, int M, int N,
                int nb, int tpc, float* __restrict__ out, long long pstride, int32_t* __restrict__ dots) {
    constexpr int W = ks_warps(FMT, BOXR), S = ks_slots(FMT, BOXR), SLOT = ks_slot(FMT, BOXR), RB = kq_bytes(FMT);
    constexpr int SA = KS_ASLOTS, WB = ks_warp_bytes(FMT, BOXR), U = BOXR / 16, MB = ks_max_boxes(BOXR);
    extern __shared__ __align__(128) uint8_t is_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    uint8_t* ring = is_smem + warp * WB;  // S weight slots, then SA activation slots
    uint8_t* aring = ring + S * SLOT;
    const uint32_t bar0 = ptx::smem_u32(is_smem + W * WB) + 8 * (S + SA) * warp;
    const uint32_t abar0 = bar0 + 8 * S;
    const int nboxes = (N + BOXR - 1) / BOXR;
    const int t0 = blockIdx.x * tpc, nt = min(tpc, nboxes - t0);  // this CTA's boxes
    // SPLIT (K split over the grid's z): this CTA's super-blocks are pz0 .. pz0 + npieces - 1,
    // its partial outputs go to slab z of `out` (pstride floats apart)
    int pz0 = 0, npieces = nb / 8;
    if constexpr (SPLIT) {
        pz0 = (int)((long long)blockIdx.z * (nb / 8) / gridDim.z);
        npieces = (int)((long long)(blockIdx.z + 1) * (nb / 8) / gridDim.z) - pz0;
        out += blockIdx.z * pstride;
    }
    const int my = warp < npieces ? (npieces - 1 - warp) / W + 1 : 0;  // this warp's pieces per box
    const int total = nt * my;
    const int m0 = blockIdx.y * 8;
    const bool h0ok = m0 + 2 * q < M, h1ok = m0 + 2 * q + 1 < M;  // the D fragment's tokens 2q, 2q + 1

    IsSchedule next{0, 0};
    auto issue = [&](int i) {  // lane 0: the copy of this warp's weight piece i into slot i % S
        const uint32_t bar = bar0 + 8 * (i % S);
        ptx::mbar_arrive_expect_tx(bar, SLOT);  // the whole box, zero-filled rows included
        ptx::tma_load_2d(ptx::smem_u32(ring + (i % S) * SLOT), &tmW, bar, (pz0 + warp + next.k * W) * (RB / 8),
                         (t0 + next.tl) * BOXR);
    };
    auto advance = [&]() {
        if (++next.tl == nt) next.tl = 0, ++next.k;
    };
    // the pass's activation rows: a box of min(8, M - m0) rows (rows past M are not copied;
    // their slot rows only ever reach outputs that are not stored)
    const bool lastp = blockIdx.y == gridDim.y - 1;
    const uint32_t abytes = (uint32_t)min(M - m0, 8) * IS_XROW;
    auto issue_acts = [&](int k) {  // lane 0: the activations of this warp's piece k into slot k % SA
        const uint32_t bar = abar0 + 8 * (k % SA);
        ptx::mbar_arrive_expect_tx(bar, abytes);
        ptx::tma_load_2d(ptx::smem_u32(aring + (k % SA) * IS_ASLOT), lastp ? &tmXl : &tmX, bar,
                         (pz0 + warp + k * W) * (IS_XROW / 8), m0);
    };
    int issued = 0, aissued = 0;
    if (lane == 0) {
        ptx::tma_prefetch_desc(&tmW);
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmXl);
        for (int i = 0; i < S + SA; ++i) ptx::mbar_init(bar0 + 8 * i, 1);
        ptx::fence_barrier_init();
    }
    __syncwarp();
    // programmatic dependent: weight pieces are requested before the previous kernel on the
    // stream has completed; the activations are read, and results written, only after.
    // Every copy queues behind the ones this SM requested before it (about 3 us deep once
    // the rings are full), and no weight piece is of use before its activations: a warp with
    // one or two pieces requests one weight piece, then its activations, then the rest; a
    // warp with more fills its weight ring first (its later pieces need the deeper ring more
    // than its first needs the earlier activations; both measured).
    const int pre = my <= 2 ? 1 : S;
    for (; issued < pre && issued < total; ++issued, advance())
        if (lane == 0) issue(issued);
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();
    for (; aissued < SA && aissued < my; ++aissued)
        if (lane == 0) issue_acts(aissued);
    for (; issued < S && issued < total; ++issued, advance())
        if (lane == 0) issue(issued);

    bool ok = true;
    int i = 0, ka = 0;  // weight and activation copies consumed
    // per box and tile of the box: rows g / g + 8, tokens (2q, 2q + 1)
    unsigned long long acc[MB][U][2];
#pragma unroll
    for (int tl = 0; tl < MB; ++tl)
#pragma unroll
        for (int u = 0; u < U; ++u) acc[tl][u][0] = acc[tl][u][1] = 0ull;
    const uint32_t msel = 0x4140u + 0x0202u * (q & 1);  // bytes 2(q & 1), 2(q & 1) + 1 of a scale word
    for (int k = 0; k < my && ok; ++k) {
        const int b0 = 8 * (pz0 + warp + k * W);  // first block of the piece
        if (!ds_wait(abar0 + 8 * (k % SA), (k / SA) & 1)) {
            ok = false;
            break;
        }
        ++ka;
        // the piece's B operands (token g, values 8q .. 8q + 7 of each block, in the k order
        // above), the f16 xd of tokens 2q, 2q + 1 per block, and the min MMA's B: the f16 xs of
        // token g in blocks 2q and 2q + 1 (k = 2q, 2q + 1, n = g)
        const uint8_t* as = aring + (k % SA) * IS_ASLOT;
        uint32_t bx[8][4], xh2[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t* cb = reinterpret_cast<const uint32_t*>(as + g * IS_XROW + j * Q8_1_BYTES + 4 + 8 * q);
            const uint32_t u0 = cb[0] ^ 0x80808080u, u1 = cb[1] ^ 0x80808080u;
            bx[j][0] = ks_code_pair(u0, 0x4240u);
            bx[j][1] = ks_code_pair(u0, 0x4341u);
            bx[j][2] = ks_code_pair(u1, 0x4240u);
            bx[j][3] = ks_code_pair(u1, 0x4341u);
            const uint32_t e0 = *reinterpret_cast<const uint32_t*>(as + 2 * q * IS_XROW + j * Q8_1_BYTES);
            const uint32_t e1 = *reinterpret_cast<const uint32_t*>(as + (2 * q + 1) * IS_XROW + j * Q8_1_BYTES);
            xh2[j] = __byte_perm(e0, e1, 0x5410);
        }
        const uint32_t xsg = __byte_perm(*reinterpret_cast<const uint32_t*>(as + g * IS_XROW + 2 * q * Q8_1_BYTES),
                                         *reinterpret_cast<const uint32_t*>(as + g * IS_XROW + (2 * q + 1) * Q8_1_BYTES),
                                         0x7632);
        // every lane holds its copy: the slot takes the piece SA ahead
        __syncwarp();
        if (aissued < my) {
            if (lane == 0) {
                ptx::fence_proxy_async_smem();
                issue_acts(aissued);
            }
            ++aissued;
        }
#pragma unroll
        for (int tl = 0; tl < MB; ++tl) {
            if (tl >= nt) break;
            if (!ds_wait(bar0 + 8 * (i % S), (i / S) & 1)) {
                ok = false;
                break;
            }
            const uint8_t* sl = ring + (i % S) * SLOT;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int n0 = (t0 + tl) * BOXR + 16 * u;
                const uint8_t* rg = sl + (16 * u + g) * RB;
                const uint8_t* rh = rg + 8 * RB;
                // Q5_K: high-bit bytes of values 8q .. 8q + 7 of rows g and g + 8 (bit j: block j)
                const uint2 qg = FMT == FMT_Q5_K ? *reinterpret_cast<const uint2*>(rg + 16 + 8 * q) : make_uint2(0u, 0u);
                const uint2 qh = FMT == FMT_Q5_K ? *reinterpret_cast<const uint2*>(rh + 16 + 8 * q) : make_uint2(0u, 0u);
                const uint4 hg = *reinterpret_cast<const uint4*>(rg), hh = *reinterpret_cast<const uint4*>(rh);
                // 6-bit sub-scales of sub-blocks 0..3 / 4..7, one per byte
                const uint32_t scg[2] = {hg.y & 0x3F3F3F3Fu, (hg.w & 0x0F0F0F0Fu) | ((hg.y >> 2) & 0x30303030u)};
                const uint32_t sch[2] = {hh.y & 0x3F3F3F3Fu, (hh.w & 0x0F0F0F0Fu) | ((hh.y >> 2) & 0x30303030u)};
                unsigned long long sg = 0ull, sh = 0ull;  // sum_j sc_j * xd_j * D_j: rows g / g + 8
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int off = kq_qs_off(FMT) + 32 * (j >> 1) + 8 * q;
                    const uint2 wg = *reinterpret_cast<const uint2*>(rg + off);
                    const uint2 wh = *reinterpret_cast<const uint2*>(rh + off);
                    constexpr uint32_t MK = 0x000F000Fu;
                    const uint32_t mk = (j & 1) ? MK << 4 : MK;
                    // A: rows g (ag) and g + 8 (ah); [0], [1]: the first MMA's k slots (2q, 2q + 1)
                    // and (2q + 8, 2q + 9); [2], [3]: the second MMA's
                    uint32_t ag[4] = {wg.x & mk, (wg.x >> 8) & mk, wg.y & mk, (wg.y >> 8) & mk};
                    uint32_t ah[4] = {wh.x & mk, (wh.x >> 8) & mk, wh.y & mk, (wh.y >> 8) & mk};
                    if constexpr (FMT == FMT_Q5_K) {
                        // the fifth bit: 16 units above a low nibble, 256 above a high one
                        const int up = (j & 1) ? 8 : 4;
                        const uint32_t bm = 0x00010001u << up;
                        ag[0] |= ((qg.x >> j) << up) & bm;
                        ag[1] |= ((qg.x >> (j + 8)) << up) & bm;
                        ag[2] |= ((qg.y >> j) << up) & bm;
                        ag[3] |= ((qg.y >> (j + 8)) << up) & bm;
                        ah[0] |= ((qh.x >> j) << up) & bm;
                        ah[1] |= ((qh.x >> (j + 8)) << up) & bm;
                        ah[2] |= ((qh.y >> j) << up) & bm;
                        ah[3] |= ((qh.y >> (j + 8)) << up) & bm;
                    }
                    float D[4];  // the block dot times 2^-24 (j even) or 2^-20 (j odd), exact
                    mma_f16_16816_z(D, ag[0], ah[0], ag[1], ah[1], bx[j][0], bx[j][1]);
                    mma_f16_16816(D, ag[2], ah[2], ag[3], ah[3], bx[j][2], bx[j][3]);
                    if constexpr (DOTS) {
                        const int b = b0 + j;
                        const float unit = (j & 1) ? 1048576.f : 16777216.f;
                        const int D0 = __float2int_rn(D[0] * unit), D1 = __float2int_rn(D[1] * unit);
                        const int D2 = __float2int_rn(D[2] * unit), D3 = __float2int_rn(D[3] * unit);
                        if (h0ok && n0 + g < N) dots[((long long)(m0 + 2 * q) * N + n0 + g) * nb + b] = D0;
                        if (h1ok && n0 + g < N) dots[((long long)(m0 + 2 * q + 1) * N + n0 + g) * nb + b] = D1;
                        if (h0ok && n0 + g + 8 < N) dots[((long long)(m0 + 2 * q) * N + n0 + g + 8) * nb + b] = D2;
                        if (h1ok && n0 + g + 8 < N) dots[((long long)(m0 + 2 * q + 1) * N + n0 + g + 8) * nb + b] = D3;
                        continue;
                    }
                    // (sc_j, sc_j) per row, sc_j / 16 for the high nibbles
                    const float cg = (j & 1) ? byte_f32_div16(scg[j >> 2], j & 3) : byte_f32(scg[j >> 2], j & 3);
                    const float ch = (j & 1) ? byte_f32_div16(sch[j >> 2], j & 3) : byte_f32(sch[j >> 2], j & 3);
                    const unsigned long long xd = is_xd2(xh2[j]);
                    sg = ptx::fma_f32x2(ptx::mul_f32x2(is_splat2(cg), xd), ptx::f2_bits(D[0], D[1]), sg);
                    sh = ptx::fma_f32x2(ptx::mul_f32x2(is_splat2(ch), xd), ptx::f2_bits(D[2], D[3]), sh);
                }
                if constexpr (!DOTS) {
                    // min term: A = m_j of rows g, g + 8 for j = 2q, 2q + 1 (sub-blocks 0..3 from
                    // the low 6 bits of scale bytes 4..7, 4..7 from bytes 8..11 and 0..3)
                    const uint32_t mwg = (q & 2) ? (((hg.w >> 4) & 0x0F0F0F0Fu) | ((hg.z >> 2) & 0x30303030u))
                                                 : (hg.z & 0x3F3F3F3Fu);
                    const uint32_t mwh = (q & 2) ? (((hh.w >> 4) & 0x0F0F0F0Fu) | ((hh.z >> 2) & 0x30303030u))
                                                 : (hh.z & 0x3F3F3F3Fu);
                    float mn[4];
                    mma_f16_1688(mn, is_byte_pair_f16(mwg, msel), is_byte_pair_f16(mwh, msel), xsg);
                    // d carries the 2^24 that undoes the weight operands' unit 2^-24
                    const float dg = f16_bits_to_f32(hg.x) * 16777216.f, ndmg = f16_bits_to_f32((hg.x >> 16) ^ 0x8000u);
                    const float dh = f16_bits_to_f32(hh.x) * 16777216.f, ndmh = f16_bits_to_f32((hh.x >> 16) ^ 0x8000u);
                    acc[tl][u][0] = ptx::fma_f32x2(is_splat2(ndmg), ptx::f2_bits(mn[0], mn[1]),
                                                   ptx::fma_f32x2(is_splat2(dg), sg, acc[tl][u][0]));
                    acc[tl][u][1] = ptx::fma_f32x2(is_splat2(ndmh), ptx::f2_bits(mn[2], mn[3]),
                                                   ptx::fma_f32x2(is_splat2(dh), sh, acc[tl][u][1]));
                }
            }
            // every lane is done with the slot: refill it with the piece S ahead
            __syncwarp();
            if (issued < total) {
                if (lane == 0) {
                    ptx::fence_proxy_async_smem();
                    issue(issued);
                }
                ++issued;
                advance();
            }
            ++i;
        }
    }
    if (!ok && lane == 0) {
        // copies still in flight must land before the CTA exits
        for (int k2 = i; k2 < issued; ++k2) {
            const uint64_t tb = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar0 + 8 * (k2 % S), (k2 / S) & 1))
                if (ptx::globaltimer_ns() - tb > DS_WAIT_LIMIT_NS) break;
        }
        for (int k2 = ka; k2 < aissued; ++k2) {
            const uint64_t tb = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(abar0 + 8 * (k2 % SA), (k2 / SA) & 1))
                if (ptx::globaltimer_ns() - tb > DS_WAIT_LIMIT_NS) break;
        }
    }
    if (DOTS) return;
    if (ok && my > 0) {
        // this warp's partial sums, [box][row][token], over its weight ring
        float* rw = reinterpret_cast<float*>(ring);
#pragma unroll
        for (int tl = 0; tl < MB; ++tl) {
            if (tl >= nt) break;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                *reinterpret_cast<unsigned long long*>(rw + (tl * BOXR + 16 * u + g) * 8 + 2 * q) = acc[tl][u][0];
                *reinterpret_cast<unsigned long long*>(rw + (tl * BOXR + 16 * u + g + 8) * 8 + 2 * q) = acc[tl][u][1];
            }
        }
    }
    if (__syncthreads_or(!ok)) return;
    const int nw = min(npieces, W);  // warps that hold partial sums
    for (int e = threadIdx.x; e < nt * BOXR * 8; e += W * 32) {
        const int tl = e / (BOXR * 8), r = (e >> 3) % BOXR, tok = e & 7;
        float v = 0.f;
        for (int w = 0; w < nw; ++w) v += reinterpret_cast<const float*>(is_smem + w * WB)[e];
        const int n = (t0 + tl) * BOXR + r;
        if (n < N && m0 + tok < M) out[(long long)(m0 + tok) * N + n] = v;
    }
}

// launch_pdl with the grid's z dimension grouped into clusters of cz CTAs (cz <= 8; the
// plain launch when cz == 1)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_zcluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                unsigned cz, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = cz;
    cfg.attrs = attr;
    cfg.numAttrs = cz > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// cluster primitives of the Q6_K stream's K split
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster arrives (release), then waits for all (acquire):
// shared-memory writes before it are visible to the cluster's reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of the same shared-memory location in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

// ------------------------------------------ Q6_K: k_mmq_q6_stream
// The tensor-core stream for Q6_K: the weights are read once, and every block dot is taken
// exactly on the tensor cores before its scales are applied ("13 . r7-r8 raw-byte MMQ
// kernel", sec. 2; "When the Product Won't Collapse", sec. "The obstruction").
// Copies.  A Q6_K row is nb/8 x 210 bytes, never a multiple of 16, so single rows cannot
// be the lines of a tensor copy; eight consecutive rows are (8 x 210 = 105 x 16).  The
// matrix is viewed as N/8 lines of eight rows, and a copy 16 lines high at byte offset
// b * row + 420 c brings, for one b in 0..7, rows b, b + 8, ..., b + 120 of a 128-row box:
// chunk c (super-blocks 2c, 2c + 1) of each, from the 16-byte boundary at or before it
// (the chunk starts 0, 4, 8 or 12 bytes into its line when K % 512 == 0).  Eight copies
// bring the box's 128 rows x one chunk; the pass's q8_1 rows for the chunk come by one
// more.  Three chunks are in flight.
// Roles.  Warp 16 issues the copies.  Once a chunk has landed, each of the 16 compute warps
// turns one of its 16 q8_1 blocks into the MMAs' B operands for all of them (the f16 codes
// in the k order below, the f32 xd pairs, and the centring terms: each sub-block's code
// sum by dp4a and two shuffles); after a hardware barrier of the 16 warps, warp w takes
// tile t = w >> 1 of the chunk: half 0 of super-block w & 1 and half 1 of the other.  (One warp converting every block
// for the others ran at a fraction of their rate and held them up: measured.)  Tile t is
// the 16 rows t, t + 8, ..., t + 120 of the box (one copy's lines, so the lanes' rows are
// 432 bytes apart: distinct banks); the two partial sums of a tile meet in shared memory
// at the end.
// Arithmetic.  Each 16-value sub-block is one m16n8k16 f16 MMA on exact operands.  A 6-bit
// code c is put together in place in an f16 half, its nibble and its two high bits
// masked and shifted into the low bits: the subnormal c x 2^-24 (for the high nibbles of
// the 128 low-bit bytes, 16 c x 2^-24, the 16 going into the sub-scale).  The MMA's
// accumulator starts from the centring term -32 x sum(u) of the sub-block's activation
// codes in the same unit (x 16 for the high nibbles).  Every partial sum is an integer
// below 2^24 units, so each sum((c - 32) u) comes out exact.  The k order inside a
// sub-block: thread (g, q) holds values 4q .. 4q + 3, k slots (2q, 2q + 1) taking values
// (4q, 4q + 2) and slots (2q + 8, 2q + 9) values (4q + 1, 4q + 3), on both sides.  Rescale
// in f32 pairs over the thread's two tokens: S += (xd, xd') (sc_a D_a + sc_b D_b) per block, then per
// super-block acc += d 2^24 S.  The odd super-block of a chunk starts 2 bytes past a
// 4-byte boundary: its words are put together from two aligned ones.
// Small outputs split K over the CTAs of a cluster (grid z); their partial tiles are
// added in rank order through distributed shared memory.  Needs K % 512 == 0, N % 8 == 0.
constexpr int Q6S_TILES = 8;                          // 16-row tiles per box: 128 rows
constexpr int Q6S_LINES = 2 * Q6S_TILES;              // eight-row lines per box
constexpr int Q6S_CW = 2 * Q6S_TILES;                 // consumer warps
constexpr int Q6S_THREADS = (Q6S_CW + 1) * 32;        // + the copy warp
constexpr int Q6S_SLOTS = 3;
constexpr int Q6S_CHUNK = 2 * Q6_K_BYTES;             // a row's bytes in one chunk: 420
constexpr int Q6S_LB = 432;                           // bytes per line of a copy: the chunk and up to 12 before it
constexpr int Q6S_COPY = Q6S_LINES * Q6S_LB;          // 6912
constexpr int Q6S_WBYTES = 8 * Q6S_COPY;              // 55296
constexpr int Q6S_XROW = 2 * IS_XROW;                 // a token's 16 q8_1 blocks of one chunk: 576
constexpr int Q6S_ABYTES = 8 * Q6S_XROW;              // 4608
constexpr int Q6S_CBLK = 32 * 16 + 4 * 16 + 4 * 8 + 16;  // per block: B operands, centring terms, xd pairs, pad
constexpr int Q6S_CBYTES = 16 * Q6S_CBLK;             // 9728
constexpr int Q6S_SLOT = Q6S_WBYTES + Q6S_ABYTES + Q6S_CBYTES;
constexpr int Q6S_SMEM = Q6S_SLOTS * Q6S_SLOT + 2 * 8 * Q6S_SLOTS;  // + the full / empty barriers
static_assert(Q6S_COPY % 128 == 0 && Q6S_SLOT % 128 == 0 && (Q6S_WBYTES + Q6S_ABYTES) % 16 == 0 &&
                  Q6S_CBLK % 16 == 0 && Q6S_LB % 16 == 0 && Q6S_LB >= Q6S_CHUNK + 12,
              "aligned regions");
static_assert(Q6S_SMEM <= 227 * 1024, "one CTA per SM");
static_assert(2 * 8 * 128 * 4 <= Q6S_SLOT, "the partial tiles fit in a slot");

// the word at byte x of a row whose base p is 4-byte aligned (MIS false) or 2 bytes past
// a 4-byte boundary (MIS true)
template <bool MIS>
__device__ __forceinline__ uint32_t q6s_word(const uint8_t* p, int x) {
    if constexpr (MIS) {
        const uint32_t lo = *reinterpret_cast<const uint32_t*>(p + x - 2);
        const uint32_t hi = *reinterpret_cast<const uint32_t*>(p + x + 2);
        return __byte_perm(lo, hi, 0x5432);
    } else {
        return *reinterpret_cast<const uint32_t*>(p + x);
    }
}
template <int SH>
__device__ __forceinline__ uint32_t q6s_shift(uint32_t v) {
    if constexpr (SH >= 0)
        return v << SH;
    else
        return v >> (-SH);
}
// byte u of a word of int8 values made unsigned (+128) as the exact f32 of the int8 value
// (SIXTEENTH: a sixteenth of it): the byte in the low mantissa bits of 2^23 (2^19), then
// 2^23 + 128 (2^19 + 8) subtracted
template <bool SIXTEENTH>
__device__ __forceinline__ float q6s_scale(uint32_t w, int u) {
    if constexpr (SIXTEENTH)
        return __uint_as_float(__byte_perm(w, 0x49000000u, 0x7440 + u)) - 524296.f;
    else
        return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440 + u)) - 8388736.f;
}

// The A operands of the sub-block pair of block jj (0..3) of a 128-value half from the
// thread's words of the low-bit bytes (w0: values 4q .., w1: 16 + 4q .. of the block's
// bytes) and of the high-bit bytes (h0, h1 likewise): [sub-block][even / odd pair].
template <int JJ>
__device__ __forceinline__ void q6s_codes(uint32_t w0, uint32_t w1, uint32_t h0, uint32_t h1, uint32_t (&a)[2][2]) {
    constexpr bool HI = JJ >= 2;                          // the high nibbles: 16 c in place
    constexpr uint32_t MK = HI ? 0x00F000F0u : 0x000F000Fu;
    constexpr int UP = HI ? 8 : 4;                        // where the two high bits go
    constexpr uint32_t BM = 0x00030003u << UP;
    a[0][0] = (w0 & MK) | (q6s_shift<UP - 2 * JJ>(h0) & BM);
    a[0][1] = ((w0 >> 8) & MK) | (q6s_shift<UP - 2 * JJ - 8>(h0) & BM);
    a[1][0] = (w1 & MK) | (q6s_shift<UP - 2 * JJ>(h1) & BM);
    a[1][1] = ((w1 >> 8) & MK) | (q6s_shift<UP - 2 * JJ - 8>(h1) & BM);
}

// Block blk (0..15) of a landed chunk's activations (as: [token][16 blocks of q8_1]) turned
// into the compute warps' operands, in the converted area after the raw rows: per lane (g,
// q) token g's B operands of both sub-blocks (values 4q .. 4q + 3 and 16 + 4q ..); the
// quad's dp4a code sums give token g's centring terms, stored (lanes q = 0, 1) where a
// compute lane reads tokens 2q', 2q' + 1 together, as is token g's xd (lane q = 2); lane
// q = 3 writes the pad (one store per lane, no branch).
__device__ __forceinline__ void q6s_convert(uint8_t* as, int blk, int lane) {
    const int g = lane >> 2, q = lane & 3;
    const uint8_t* xb = as + g * Q6S_XROW + blk * Q8_1_BYTES;
    const uint32_t c0w = *reinterpret_cast<const uint32_t*>(xb + 4 + 4 * q);
    const uint32_t c1w = *reinterpret_cast<const uint32_t*>(xb + 20 + 4 * q);
    const uint32_t xdw = *reinterpret_cast<const uint32_t*>(xb);
    int s0 = __dp4a((int)c0w, 0x01010101, 0), s1 = __dp4a((int)c1w, 0x01010101, 0);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 1);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 1);
    s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
    const uint32_t u0 = c0w ^ 0x80808080u, u1 = c1w ^ 0x80808080u;
    uint4 bf;
    bf.x = ks_code_pair(u0, 0x4240u);
    bf.y = ks_code_pair(u0, 0x4341u);
    bf.z = ks_code_pair(u1, 0x4240u);
    bf.w = ks_code_pair(u1, 0x4341u);
    uint8_t* cb = as + Q6S_ABYTES + blk * Q6S_CBLK;
    *reinterpret_cast<uint4*>(cb + 16 * lane) = bf;
    // -32 x sum(u) in units of 2^-24 (x 16 for the high nibbles: blocks 2, 3 of each half)
    const float unit = (blk & 2) ? -512.f / 16777216.f : -32.f / 16777216.f;
    const float v = q == 2 ? f16_bits_to_f32(xdw) : (float)(q ? s1 : s0) * unit;
    const int off = q < 2 ? 512 + 16 * (g >> 1) + 4 * (g & 1) + 8 * q
                          : (q == 2 ? 576 + 8 * (g >> 1) + 4 * (g & 1) : 608 + 4 * (g & 3));
    *reinterpret_cast<float*>(cb + off) = v;
}

// mma_f16_16816 without the volatile qualifier: a pure function of its operands, which the
// compiler may schedule among the surrounding work (several blocks' MMAs in flight)
__device__ __forceinline__ void q6s_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Half H (blocks 4H .. 4H + 3) of one super-block of one 16-row tile: the thread's A rows g
// (bytes at pg; weight row ng) and g + 8 (ph; weight row ng + 64); cv: the converted
// activations of the super-block's eight blocks.  Accumulates into accg / acch (tokens 2q,
// 2q + 1), or, with DOTS, writes the integer block dots of blocks b0 + 4H .. b0 + 4H + 3.
template <bool MIS, bool DOTS, int H>
__device__ __forceinline__ void q6s_half(const uint8_t* pg, const uint8_t* ph, const uint8_t* cv, int lane,
                                         unsigned long long& accg, unsigned long long& acch, int32_t* dots, int M,
                                         int N, int nb, int m0, int ng, int b0) {
    const int q = lane & 3;
    uint32_t scg[2], sch[2];  // the half's 8 int8 sub-scales of each row, made unsigned
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        scg[i] = q6s_word<MIS>(pg, 192 + 8 * H + 4 * i) ^ 0x80808080u;
        sch[i] = q6s_word<MIS>(ph, 192 + 8 * H + 4 * i) ^ 0x80808080u;
    }
    unsigned long long sg = 0ull, sh = 0ull;
    const uint32_t hg0 = q6s_word<MIS>(pg, 128 + 32 * H + 4 * q), hg1 = q6s_word<MIS>(pg, 144 + 32 * H + 4 * q);
    const uint32_t hh0 = q6s_word<MIS>(ph, 128 + 32 * H + 4 * q), hh1 = q6s_word<MIS>(ph, 144 + 32 * H + 4 * q);
#pragma unroll
    for (int jo = 0; jo < 2; ++jo) {
        const uint32_t wg0 = q6s_word<MIS>(pg, 64 * H + 32 * jo + 4 * q);
        const uint32_t wg1 = q6s_word<MIS>(pg, 64 * H + 32 * jo + 16 + 4 * q);
        const uint32_t wh0 = q6s_word<MIS>(ph, 64 * H + 32 * jo + 4 * q);
        const uint32_t wh1 = q6s_word<MIS>(ph, 64 * H + 32 * jo + 16 + 4 * q);
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            const int jj = jo + 2 * hi, blk = 4 * H + jj;
            uint32_t ag[2][2], ah[2][2];
            if (jj == 0) {
                q6s_codes<0>(wg0, wg1, hg0, hg1, ag);
                q6s_codes<0>(wh0, wh1, hh0, hh1, ah);
            } else if (jj == 1) {
                q6s_codes<1>(wg0, wg1, hg0, hg1, ag);
                q6s_codes<1>(wh0, wh1, hh0, hh1, ah);
            } else if (jj == 2) {
                q6s_codes<2>(wg0, wg1, hg0, hg1, ag);
                q6s_codes<2>(wh0, wh1, hh0, hh1, ah);
            } else {
                q6s_codes<3>(wg0, wg1, hg0, hg1, ag);
                q6s_codes<3>(wh0, wh1, hh0, hh1, ah);
            }
            const uint8_t* cb = cv + blk * Q6S_CBLK;
            const uint4 bf = *reinterpret_cast<const uint4*>(cb + 16 * lane);
            const float4 bz = *reinterpret_cast<const float4*>(cb + 512 + 16 * q);
            float D0[4] = {bz.x, bz.y, bz.x, bz.y}, D1[4] = {bz.z, bz.w, bz.z, bz.w};
            q6s_mma(D0, ag[0][0], ah[0][0], ag[0][1], ah[0][1], bf.x, bf.y);
            q6s_mma(D1, ag[1][0], ah[1][0], ag[1][1], ah[1][1], bf.z, bf.w);
            const int s0 = 2 * jj, s1 = 2 * jj + 1;  // the block's sub-blocks among the half's 8
            if constexpr (DOTS) {
                const float unit = hi ? 1048576.f : 16777216.f;
                const int cg0 = (int)((scg[s0 >> 2] >> (8 * (s0 & 3))) & 0xFFu) - 128;
                const int cg1 = (int)((scg[s1 >> 2] >> (8 * (s1 & 3))) & 0xFFu) - 128;
                const int ch0 = (int)((sch[s0 >> 2] >> (8 * (s0 & 3))) & 0xFFu) - 128;
                const int ch1 = (int)((sch[s1 >> 2] >> (8 * (s1 & 3))) & 0xFFu) - 128;
                const int v[4] = {cg0 * __float2int_rn(D0[0] * unit) + cg1 * __float2int_rn(D1[0] * unit),
                                  cg0 * __float2int_rn(D0[1] * unit) + cg1 * __float2int_rn(D1[1] * unit),
                                  ch0 * __float2int_rn(D0[2] * unit) + ch1 * __float2int_rn(D1[2] * unit),
                                  ch0 * __float2int_rn(D0[3] * unit) + ch1 * __float2int_rn(D1[3] * unit)};
                const int b = b0 + blk;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = m0 + 2 * q + (e & 1), n = ng + 64 * (e >> 1);
                    if (m < M && n < N) dots[((long long)m * N + n) * nb + b] = v[e];
                }
            } else {
                const float cg0 = hi ? q6s_scale<true>(scg[s0 >> 2], s0 & 3) : q6s_scale<false>(scg[s0 >> 2], s0 & 3);
                const float cg1 = hi ? q6s_scale<true>(scg[s1 >> 2], s1 & 3) : q6s_scale<false>(scg[s1 >> 2], s1 & 3);
                const float ch0 = hi ? q6s_scale<true>(sch[s0 >> 2], s0 & 3) : q6s_scale<false>(sch[s0 >> 2], s0 & 3);
                const float ch1 = hi ? q6s_scale<true>(sch[s1 >> 2], s1 & 3) : q6s_scale<false>(sch[s1 >> 2], s1 & 3);
                const unsigned long long xd = *reinterpret_cast<const unsigned long long*>(cb + 576 + 8 * q);
                const unsigned long long tg = ptx::fma_f32x2(
                    is_splat2(cg1), ptx::f2_bits(D1[0], D1[1]), ptx::mul_f32x2(is_splat2(cg0), ptx::f2_bits(D0[0], D0[1])));
                const unsigned long long th = ptx::fma_f32x2(
                    is_splat2(ch1), ptx::f2_bits(D1[2], D1[3]), ptx::mul_f32x2(is_splat2(ch0), ptx::f2_bits(D0[2], D0[3])));
                sg = ptx::fma_f32x2(xd, tg, sg);
                sh = ptx::fma_f32x2(xd, th, sh);
            }
        }
    }
    if constexpr (!DOTS) {
        // d carries the 2^24 that undoes the weight operands' unit 2^-24
        const uint32_t dwg = MIS ? (*reinterpret_cast<const uint32_t*>(pg + 206) >> 16)
                                 : *reinterpret_cast<const uint32_t*>(pg + 208);
        const uint32_t dwh = MIS ? (*reinterpret_cast<const uint32_t*>(ph + 206) >> 16)
                                 : *reinterpret_cast<const uint32_t*>(ph + 208);
        accg = ptx::fma_f32x2(is_splat2(f16_bits_to_f32(dwg) * 16777216.f), sg, accg);
        acch = ptx::fma_f32x2(is_splat2(f16_bits_to_f32(dwh) * 16777216.f), sh, acch);
    }
}

// hardware barrier 1 of the CTA over the compute warps, returning whether any of them
// arrived with p set (every warp sees the same answer)
__device__ __forceinline__ bool q6s_bar_any(bool p) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred a, b;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred b, 1, %2, a;\n selp.u32 %0, 1, 0, b;\n}"
        : "=r"(r)
        : "r"((uint32_t)p), "n"(Q6S_CW * 32)
        : "memory");
    return r != 0;
}
// one thread's bounded wait on an mbarrier phase, backing off between polls
__device__ __forceinline__ bool q6s_wait1(uint32_t bar, uint32_t parity) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        __nanosleep(128);
        if (ptx::globaltimer_ns() - t0 > DS_WAIT_LIMIT_NS) {
            atomicOr(&g_small_error, ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

template <bool DOTS, bool GSPLIT = false>
__global__ void __launch_bounds__(Q6S_THREADS, 1)
k_mmq_q6_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmXl, int M, int N, int nb, unsigned stagger_ns,
                float* __restrict__ out, long long pstride, int32_t* __restrict__ dots) {
    extern __shared__ __align__(128) uint8_t is_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const uint32_t full0 = ptx::smem_u32(is_smem + Q6S_SLOTS * Q6S_SLOT);
    const uint32_t empty0 = full0 + 8 * Q6S_SLOTS;
    const int nsb = nb / 8, nch = nsb / 2;
    const long long rowb = (long long)nsb * Q6_K_BYTES;  // bytes per weight row
    const int box = blockIdx.x, m0 = blockIdx.y * 8;
    const int splits = gridDim.z, z = blockIdx.z;
    const int c0 = (int)((long long)z * nch / splits), nmy = (int)((long long)(z + 1) * nch / splits) - c0;
    const bool lastp = blockIdx.y == gridDim.y - 1;
    const uint32_t abytes = (uint32_t)min(M - m0, 8) * Q6S_XROW;
    const int CP = Q6S_CW;  // the copy warp
    auto issue_w = [&](int i) {  // lane 0 of the copy warp: the weights of chunk c0 + i
        const int sl = i % Q6S_SLOTS;
        const uint32_t dst = ptx::smem_u32(is_smem + sl * Q6S_SLOT), bar = full0 + 8 * sl;
        const long long cb = (long long)Q6S_CHUNK * (c0 + i);
#pragma unroll 1
        for (int b = 0; b < 8; ++b)
            ptx::tma_load_2d(dst + b * Q6S_COPY, &tmW, bar, (int)(((b * rowb + cb) & ~15ll) >> 3), box * Q6S_LINES);
    };
    auto issue_x = [&](int i) {  // the pass's activation rows of chunk c0 + i
        const int sl = i % Q6S_SLOTS;
        ptx::tma_load_2d(ptx::smem_u32(is_smem + sl * Q6S_SLOT + Q6S_WBYTES), lastp ? &tmXl : &tmX, full0 + 8 * sl,
                         (c0 + i) * (Q6S_XROW / 8), m0);
    };
    const int pre = min(nmy, Q6S_SLOTS);
    if (threadIdx.x == 0) {
        for (int i = 0; i < Q6S_SLOTS; ++i) {
            ptx::mbar_init(full0 + 8 * i, 1);
            ptx::mbar_init(empty0 + 8 * i, Q6S_CW);
        }
        ptx::fence_barrier_init();
    }
    __syncthreads();
    // programmatic dependent: the first weight chunk is requested before the previous kernel
    // on the stream has completed; activations are read, and results written, after
    uint64_t t_first = 0;
    if (warp == CP && lane == 0) {
        ptx::tma_prefetch_desc(&tmW);
        ptx::tma_prefetch_desc(&tmX);
        ptx::tma_prefetch_desc(&tmXl);
        if (nmy > 0) {
            ptx::mbar_arrive_expect_tx(full0, Q6S_WBYTES + abytes);
            issue_w(0);
            t_first = ptx::globaltimer_ns();
        }
    }
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();

    bool ok = true;
    unsigned long long accg = 0ull, acch = 0ull;  // rows g / g + 8 of the warp's tile, tokens (2q, 2q + 1)
    if (warp == CP) {
        if (lane == 0) {
            // the ring's first chunks one stagger apart (about one chunk's transfer time at
            // the GPU's bandwidth share of this CTA), or as soon as the one before has landed:
            // requested together, they arrive interleaved and the first lands only with the last
            if (nmy > 0) issue_x(0);
            for (int i = 1; i < pre; ++i) {
                const uint64_t due = t_first + (uint64_t)i * stagger_ns;
                while (ptx::globaltimer_ns() < due && !ptx::mbar_test_wait(full0 + 8 * (i - 1), 0)) __nanosleep(64);
                ptx::mbar_arrive_expect_tx(full0 + 8 * i, Q6S_WBYTES + abytes);
                issue_w(i);
                issue_x(i);
            }
            int issued = pre;
            for (int i = pre; i < nmy; ++i, ++issued) {
                const int sl = i % Q6S_SLOTS;
                if (!q6s_wait1(empty0 + 8 * sl, (i / Q6S_SLOTS - 1) & 1)) {
                    ok = false;
                    break;
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive_expect_tx(full0 + 8 * sl, Q6S_WBYTES + abytes);
                issue_w(i);
                issue_x(i);
            }
            if (!ok) {
            // copies still in flight must land before the CTA exits
                for (int k = max(0, issued - Q6S_SLOTS); k < issued; ++k) {
                    const uint64_t tb = ptx::globaltimer_ns();
                    while (!ptx::mbar_try_wait(full0 + 8 * (k % Q6S_SLOTS), (k / Q6S_SLOTS) & 1))
                        if (ptx::globaltimer_ns() - tb > DS_WAIT_LIMIT_NS) break;
                }
            }
        }
    } else {
        const int t = warp >> 1, j = warp & 1;
        const int ng = box * 128 + 8 * g + t;  // the weight row of the thread's first A row
        // where the tile's rows start in their lines: (t * row + 420 c) mod 16, 0, 4, 8 or 12
        const int rb16 = (int)(rowb & 15);
        for (int i = 0; i < nmy; ++i) {
            const int sl = i % Q6S_SLOTS;
            // each compute warp converts one block of the landed chunk; the barrier then has
            // every block converted, and tells every warp whether any wait ran out (a lone
            // warp leaving the loop would leave the others at the barrier)
            const bool landed = ds_wait(full0 + 8 * sl, (i / Q6S_SLOTS) & 1);
            if (landed) q6s_convert(is_smem + sl * Q6S_SLOT + Q6S_WBYTES, warp, lane);
            if (q6s_bar_any(!landed)) {
                ok = false;
                break;
            }
            const int c = c0 + i;
            const uint8_t* slot = is_smem + sl * Q6S_SLOT;
            const int o = (t * rb16 + 4 * c) & 15;
            // super-block 0 of the chunk (4-byte aligned) and super-block 1 (2 bytes past):
            // warp j takes half 0 of super-block j and half 1 of the other, so that every
            // warp does one aligned and one misaligned half (equal work at the barrier)
            const uint8_t* p0 = slot + t * Q6S_COPY + g * Q6S_LB + o;
            const uint8_t* p1 = p0 + Q6_K_BYTES;
            const uint8_t* cv0 = slot + Q6S_WBYTES + Q6S_ABYTES;
            const uint8_t* cv1 = cv0 + 8 * Q6S_CBLK;
            const int b00 = 16 * c, b01 = 16 * c + 8;
            const int L8 = 8 * Q6S_LB;
            if (j) {
                q6s_half<true, DOTS, 0>(p1, p1 + L8, cv1, lane, accg, acch, dots, M, N, nb, m0, ng, b01);
                q6s_half<false, DOTS, 1>(p0, p0 + L8, cv0, lane, accg, acch, dots, M, N, nb, m0, ng, b00);
            } else {
                q6s_half<false, DOTS, 0>(p0, p0 + L8, cv0, lane, accg, acch, dots, M, N, nb, m0, ng, b00);
                q6s_half<true, DOTS, 1>(p1, p1 + L8, cv1, lane, accg, acch, dots, M, N, nb, m0, ng, b01);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(empty0 + 8 * sl);
        }
    }
    const bool bad = __syncthreads_or(!ok);
    // the tile's two partial sums ([super-block parity][token][128 rows] over slot 0), then
    // their sum in place; every copy has landed by now
    float* red = reinterpret_cast<float*>(is_smem);
    if (!DOTS && !bad && warp < Q6S_CW) {
        const int t = warp >> 1, j = warp & 1, r = 8 * g + t;  // box rows r and r + 64
        float* rj = red + j * 1024;
        rj[(2 * q) * 128 + r] = __uint_as_float((uint32_t)accg);
        rj[(2 * q + 1) * 128 + r] = __uint_as_float((uint32_t)(accg >> 32));
        rj[(2 * q) * 128 + r + 64] = __uint_as_float((uint32_t)acch);
        rj[(2 * q + 1) * 128 + r + 64] = __uint_as_float((uint32_t)(acch >> 32));
    }
    __syncthreads();
    if (!DOTS && !bad)
        for (int e = threadIdx.x; e < 1024; e += Q6S_THREADS) red[e] += red[1024 + e];
    if (!GSPLIT && splits > 1) {
        // the cluster's CTAs (ranks 0 .. splits - 1 in K order) hold partial tiles; rank 0
        // adds them in rank order and stores; nobody leaves while its tile may be read
        cluster_sync();
        if (!DOTS && !bad && cluster_ctarank() == 0) {
            const uint32_t base = ptx::smem_u32(red);
            for (int e = threadIdx.x; e < 1024; e += Q6S_THREADS) {
                const int tok = e >> 7, n = box * 128 + (e & 127);
                float v = 0.f;
                for (int r = 0; r < splits; ++r) v += ld_cluster_f32(cluster_map(base + 4 * e, r));
                if (n < N && m0 + tok < M) out[(long long)(m0 + tok) * N + n] = v;
            }
        }
        cluster_sync();
    } else {
        // the whole K, or (GSPLIT: a split over the grid's z without clusters) this CTA's
        // partial tile to slab z of `out`, pstride floats apart
        __syncthreads();
        if (GSPLIT) out += z * pstride;
        if (!DOTS && !bad)
            for (int e = threadIdx.x; e < 1024; e += Q6S_THREADS) {
                const int tok = e >> 7, n = box * 128 + (e & 127);
                if (n < N && m0 + tok < M) out[(long long)(m0 + tok) * N + n] = red[e];
            }
    }
}

// the activation maps of the streams: 8-row boxes for the full passes, and for the last pass
// a box of its own rows (M - 8 (passes - 1)); copying rows past M as the copy engine's
// zero fill was measured to slow a one-row pass down by a third
inline bool make_act_maps(CUtensorMap* tx, CUtensorMap* txl, const uint8_t* x8, int64_t M, int nb,
                          uint32_t box_bytes = IS_XROW) {
    const uint32_t last = (uint32_t)(M - 8 * ((M - 1) / 8));
    return make_byte_map(tx, x8, (uint64_t)nb * Q8_1_BYTES, (uint64_t)M, box_bytes, 8, 8) &&
           make_byte_map(txl, x8, (uint64_t)nb * Q8_1_BYTES, (uint64_t)M, box_bytes, last, 8);
}

// boxes per CTA: the fewest (at most max_boxes) that keep the grid within the two CTAs per
// SM that are resident at once (no second, partial wave)
inline int64_t stream_tpc(int64_t nboxes, int max_boxes) {
    const int64_t per_wave = 2 * (int64_t)device_shape().sms;
    const int64_t tpc = (nboxes + per_wave - 1) / per_wave;
    return tpc < 1 ? 1 : (tpc > max_boxes ? max_boxes : tpc);
}

// ------------------------------------------ K splits of the i8 / kq streams
// A stream grid whose CTAs would load the SMs unevenly, or that needs a second wave, takes
// z K splits (grid z) and, with them, tpc boxes per CTA: 3584 x 18944 through eight rows is
// 224 one-box CTAs on 152 SMs, 72 SMs with two boxes and 80 with one; through sixteen rows,
// 448 CTAs in two waves.  Each split writes its partial outputs to a slab of scratch and
// k_stream_ksum adds the slabs in the order z = 0, 1, ... (the same order at every call, so
// the output is deterministic).  Cost of a grid: its waves (two CTAs per SM resident) x
// (KS_START + a CTA's pieces, tpc boxes x ceil(pieces / z)), KS_START pieces standing for a
// CTA's start-up (~5 us, the first activations landing behind the SM's queued weight
// copies, against ~0.17 us a piece).  The cheapest one-wave grid that leaves each warp two
// pieces or more is taken where it saves more than 15 %; grids of several passes only for
// a long K (32 pieces or more, the measured range).  Measured (Q4_K, graph replays):
// 3584 x 18944, eight rows: 16.3 us unsplit, 13.25 with 3 boxes x 4 splits on 300 CTAs
// (57 pieces a CTA), 19.2 with 3 x 2 on 150 (111 pieces, one CTA per SM), 15.2 with 2 x 2
// or 4 x 4 (74 / 76), 18.5 with 4 x 8 (two waves); sixteen rows 25.6 -> 20.9 (3 x 2),
// Q8_0 32.8 -> 24.7; 24 rows 39.2 -> 34.9 (3 boxes, no split); 4096 x 14336, sixteen rows,
// 23.9 -> 19.4 (2 boxes, no split); 512 x 18944, eight rows, 11.0 -> 5.5 (4 splits).
// Outside stream capture a split call costs the host about 14 us (the second launch, the
// scratch calls), more than the GPU time it saves on small weights: eager calls split only
// weights of 32 MB and more (back to back, 512 x 18944 Q4_K 11.3 -> 13.9 us split, 3584 x
// 18944 16.7 -> 14.5); smaller ones may still take more boxes per CTA, unsplit.
std::atomic<int> g_small_ksplit{0};  // test switches: splits (0: the rule) and boxes per CTA (0: the launcher's)
std::atomic<int> g_small_kboxes{0};
constexpr int64_t KS_START = 30;

struct StreamGrid {
    int64_t tpc;
    int z;
};

constexpr int64_t EAGER_SPLIT_MIN_BYTES = (int64_t)32 << 20;

// true when `s` is being captured (a split's host cost is then paid once, at capture)
inline bool stream_captured(cudaStream_t s) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs != cudaStreamCaptureStatusNone;
}

inline StreamGrid stream_grid(int64_t nboxes, int max_boxes, int64_t passes, int64_t pieces, int warps,
                              int64_t wbytes, cudaStream_t s) {
    const int64_t base = stream_tpc(nboxes, max_boxes);
    const int forced = g_small_ksplit.load(), fboxes = g_small_kboxes.load();
    if (forced > 0)
        return {fboxes > 0 ? std::min<int64_t>(fboxes, max_boxes) : base,
                (int)std::min<int64_t>(forced, std::max<int64_t>(pieces, 1))};
    if (passes != 1 && pieces < 32) return {base, 1};
    const int zmax = wbytes < EAGER_SPLIT_MIN_BYTES && !stream_captured(s) ? 1 : 8;
    const int64_t slots = 2 * (int64_t)device_shape().sms;
    auto ctas = [&](int64_t t, int64_t z) { return (nboxes + t - 1) / t * z * passes; };
    auto cost = [&](int64_t t, int64_t z) {
        return (ctas(t, z) + slots - 1) / slots * (KS_START + t * ((pieces + z - 1) / z));
    };
    StreamGrid best{base, 1};
    for (int z = 1; z <= zmax && (z == 1 || pieces >= 2LL * warps * z); ++z)
        for (int64_t t = 1; t <= max_boxes; ++t)
            if (ctas(t, z) <= slots && cost(t, z) < cost(best.tpc, best.z)) best = {t, z};
    return cost(best.tpc, best.z) * 20 < cost(base, 1) * 17 ? best : StreamGrid{base, 1};
}

// slab 0 + slab 1 + ... of a split stream's partial outputs, as a programmatic dependent of
// the stream kernel; it releases the next kernel on the stream before its own wait (that
// kernel's wait still covers this one's stores)
__global__ void __launch_bounds__(256) k_stream_ksum(const float* __restrict__ part, int splits, long long pstride,
                                                     long long n, float* __restrict__ out) {
    ptx::grid_dep_launch_dependents();
    ptx::grid_dep_wait();
    for (long long i = blockIdx.x * 256LL + threadIdx.x; i < n; i += gridDim.x * 256LL) {
        float v = __ldcs(part + i);
        for (int z = 1; z < splits; ++z) v += __ldcs(part + z * pstride + i);
        out[i] = v;
    }
}

// Scratch for the partial outputs.  Outside stream capture: the library's stream-ordered
// pool, allocated and freed on the call's stream like every other call's scratch.  Under
// capture, the allocation is a root node of the graph with one edge, into the stream
// kernel's node, and the free a leaf node after the sum: captured in stream order the two
// would sit between this call's kernels and its neighbours' and end the programmatic
// overlap of consecutive calls (measured ~4 us a call).
struct SplitScratch {
    float* p = nullptr;
    cudaGraph_t graph = nullptr;  // set under capture
    cudaGraphNode_t alloc = nullptr;
};

int split_scratch_alloc(size_t bytes, cudaStream_t s, SplitScratch* ss, const char* fn) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaGraph_t g = nullptr;
    if (cudaStreamGetCaptureInfo(s, &cs, nullptr, &g) != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_CUDA, "cudaStreamGetCaptureInfo failed");
        return MMQ_ERR_CUDA;
    }
    if (cs == cudaStreamCaptureStatusNone) {
        void* p = nullptr;
        const int st = scratch_alloc(bytes, s, &p, fn);
        ss->p = static_cast<float*>(p);
        return st;
    }
    int dev = 0;
    cudaMemAllocNodeParams prm = {};
    prm.poolProps.allocType = cudaMemAllocationTypePinned;
    prm.poolProps.location.type = cudaMemLocationTypeDevice;
    prm.bytesize = bytes;
    if (cs != cudaStreamCaptureStatusActive || cudaGetDevice(&dev) != cudaSuccess ||
        (prm.poolProps.location.id = dev, cudaGraphAddMemAllocNode(&ss->alloc, g, nullptr, 0, &prm)) != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_NOMEM, "scratch allocation node for the K split failed");
        return MMQ_ERR_NOMEM;
    }
    ss->p = static_cast<float*>(prm.dptr);
    ss->graph = g;
    return MMQ_OK;
}

// under capture, right after the stream kernel's launch (the stream's one dependency is
// then that kernel's node): the node depends on the allocation
int split_scratch_bind(const SplitScratch& ss, cudaStream_t s, const char* fn) {
    if (!ss.graph) return MMQ_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t* deps = nullptr;
    const cudaGraphEdgeData* edata = nullptr;
    size_t nd = 0;
    if (cudaStreamGetCaptureInfo(s, &cs, nullptr, nullptr, &deps, &edata, &nd) != cudaSuccess || nd != 1 ||
        cudaGraphAddDependencies(ss.graph, &ss.alloc, deps, nullptr, 1) != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_CUDA, "ordering the K split's scratch in the captured graph failed");
        return MMQ_ERR_CUDA;
    }
    return MMQ_OK;
}

void split_scratch_free(const SplitScratch& ss, cudaStream_t s) {
    if (!ss.p) return;
    if (!ss.graph) {
        scratch_free(ss.p, s);
        return;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t* deps = nullptr;
    const cudaGraphEdgeData* edata = nullptr;
    size_t nd = 0;
    cudaGraphNode_t fnode = nullptr;
    if (cudaStreamGetCaptureInfo(s, &cs, nullptr, nullptr, &deps, &edata, &nd) != cudaSuccess ||
        cudaGraphAddMemFreeNode(&fnode, ss.graph, deps, nd, ss.p) != cudaSuccess)
        cudaGetLastError();
}

// A stream kernel's launch with z K splits: launch(out, pstride, z) launches it (with its
// profiling scope) into `out` or the partial slabs and returns its status; the sum follows.
template <typename Launch>
int launch_stream_split(int z, int64_t M, int64_t N, float* out, cudaStream_t s, const char* fn, Launch&& launch,
                        SplitScratch* ss) {
    if (z <= 1) return launch(out, 0LL, 1u);
    const long long pstride = (M * N + 63) / 64 * 64;  // 256-byte slabs
    int st = split_scratch_alloc((size_t)z * pstride * sizeof(float), s, ss, fn);
    if (st != MMQ_OK) return st;
    st = launch(ss->p, pstride, (unsigned)z);
    if (st == MMQ_OK) {
        const long long n = M * N;
        const unsigned blocks = (unsigned)std::min<long long>((n + 255) / 256, 4LL * device_shape().sms);
        ProfScope ps("k_stream_ksum", s);
        st = pdl_status(launch_pdl(k_stream_ksum, dim3(blocks), dim3(256), 0, s, (const float*)ss->p, z, pstride, n, out),
                        fn);
    }
    split_scratch_free(*ss, s);
    return st;
}

int launch_i8_stream_q8_0(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                          int32_t* dots, cudaStream_t s, const char* fn) {
    const int64_t ntiles = (N + 15) / 16;
    const StreamGrid sg = dots ? StreamGrid{stream_tpc(ntiles, IS_MAX_TPC), 1}
                               : stream_grid(ntiles, IS_MAX_TPC, (M + 7) / 8, nb / 8, IS_WARPS,
                                             N * (int64_t)nb * Q8_0_BYTES, s);
    const int64_t tpc = sg.tpc;
    static SmemAttr attr, attr_d, attr_s;
    const int e = dots       ? ensure_smem((const void*)k_mmq_i8_stream<true>, I8_SMEM, attr_d)
                  : sg.z > 1 ? ensure_smem((const void*)k_mmq_i8_stream<false, true>, I8_SMEM, attr_s)
                             : ensure_smem((const void*)k_mmq_i8_stream<false>, I8_SMEM, attr);
    if (e != MMQ_OK) {
        report(fn, e, "shared-memory request refused");
        return e;
    }
    CUtensorMap tw, tx, txl;
    if (!make_byte_map(&tw, w8, (uint64_t)nb * Q8_0_BYTES, (uint64_t)N, 8 * Q8_0_BYTES, 16, 8) ||
        !make_act_maps(&tx, &txl, x8, M, nb)) {
        report(fn, MMQ_ERR_CUDA, "tensor map encoding failed");
        return MMQ_ERR_CUDA;
    }
    const dim3 grid((unsigned)((ntiles + tpc - 1) / tpc), (unsigned)((M + 7) / 8));
    const int z = sg.z;
    SplitScratch ss;
    return launch_stream_split(
        z, M, N, out, s, fn,
        [&](float* o, long long pstride, unsigned gz) {
            ProfScope ps("k_mmq_i8_stream", s);
            const dim3 g3(grid.x, grid.y, gz);
            const dim3 blk(IS_WARPS * 32);
            const int st = pdl_status(
                dots     ? launch_pdl(k_mmq_i8_stream<true>, g3, blk, (size_t)I8_SMEM, s, tw, tx, txl, (int)M, (int)N, nb,
                                      (int)tpc, o, pstride, dots)
                : gz > 1 ? launch_pdl(k_mmq_i8_stream<false, true>, g3, blk, (size_t)I8_SMEM, s, tw, tx, txl, (int)M,
                                      (int)N, nb, (int)tpc, o, pstride, dots)
                         : launch_pdl(k_mmq_i8_stream<false>, g3, blk, (size_t)I8_SMEM, s, tw, tx, txl, (int)M, (int)N,
                                      nb, (int)tpc, o, pstride, dots),
                fn);
            return st == MMQ_OK ? split_scratch_bind(ss, s, fn) : st;
        },
        &ss);
}

template <int FMT, int BOXR>
int launch_kq_stream_b(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                       int32_t* dots, cudaStream_t s, const char* fn) {
    const int64_t nboxes = (N + BOXR - 1) / BOXR;
    const StreamGrid sg = dots ? StreamGrid{stream_tpc(nboxes, ks_max_boxes(BOXR)), 1}
                               : stream_grid(nboxes, ks_max_boxes(BOXR), (M + 7) / 8, nb / 8, ks_warps(FMT, BOXR),
                                             N * (int64_t)(nb / 8) * kq_bytes(FMT), s);
    const int64_t tpc = sg.tpc;
    constexpr int smem = ks_smem_bytes(FMT, BOXR);
    static SmemAttr attr, attr_d, attr_s;
    const int e = dots       ? ensure_smem((const void*)k_mmq_kq_stream<FMT, BOXR, true>, smem, attr_d)
                  : sg.z > 1 ? ensure_smem((const void*)k_mmq_kq_stream<FMT, BOXR, false, true>, smem, attr_s)
                             : ensure_smem((const void*)k_mmq_kq_stream<FMT, BOXR, false>, smem, attr);
    if (e != MMQ_OK) {
        report(fn, e, "shared-memory request refused");
        return e;
    }
    CUtensorMap tw, tx, txl;
    if (!make_byte_map(&tw, w8, (uint64_t)(nb / 8) * kq_bytes(FMT), (uint64_t)N, kq_bytes(FMT), BOXR, 8) ||
        !make_act_maps(&tx, &txl, x8, M, nb)) {
        report(fn, MMQ_ERR_CUDA, "tensor map encoding failed");
        return MMQ_ERR_CUDA;
    }
    const dim3 grid((unsigned)((nboxes + tpc - 1) / tpc), (unsigned)((M + 7) / 8));
    const dim3 block(ks_warps(FMT, BOXR) * 32);
    const int z = sg.z;
    SplitScratch ss;
    return launch_stream_split(
        z, M, N, out, s, fn,
        [&](float* o, long long pstride, unsigned gz) {
            ProfScope ps("k_mmq_kq_stream", s);
            const dim3 g3(grid.x, grid.y, gz);
            const int st = pdl_status(
                dots     ? launch_pdl(k_mmq_kq_stream<FMT, BOXR, true>, g3, block, (size_t)smem, s, tw, tx, txl, (int)M,
                                      (int)N, nb, (int)tpc, o, pstride, dots)
                : gz > 1 ? launch_pdl(k_mmq_kq_stream<FMT, BOXR, false, true>, g3, block, (size_t)smem, s, tw, tx, txl,
                                      (int)M, (int)N, nb, (int)tpc, o, pstride, dots)
                         : launch_pdl(k_mmq_kq_stream<FMT, BOXR, false>, g3, block, (size_t)smem, s, tw, tx, txl,
                                      (int)M, (int)N, nb, (int)tpc, o, pstride, dots),
                fn);
            return st == MMQ_OK ? split_scratch_bind(ss, s, fn) : st;
        },
        &ss);
}

// 32-row boxes when there are at least two of them per SM, else 16-row boxes
template <int FMT>
int launch_kq_stream(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out, int32_t* dots,
                     cudaStream_t s, const char* fn) {
    if ((N + 31) / 32 >= 2 * (int64_t)device_shape().sms)
        return launch_kq_stream_b<FMT, 32>(x8, w8, M, N, nb, out, dots, s, fn);
    return launch_kq_stream_b<FMT, 16>(x8, w8, M, N, nb, out, dots, s, fn);
}

// the Q6_K tensor-core stream takes K % 512 == 0 (chunks of two super-blocks start 4-byte
// aligned), N % 8 == 0 (the matrix as lines of eight rows) and lines below 2 GB
bool q6_stream_fits(int64_t N, int nb) {
    return nb % 16 == 0 && N % 8 == 0 && (int64_t)(nb / 8) * 8 * Q6_K_BYTES < ((int64_t)1 << 31);
}

// K split over clusters of 2, 4 or 8 CTAs while the grid still fits the SMs at one CTA each
// (powers of two: clusters pack into the GPCs without leaving SMs over)
int q6_stream_splits(int64_t boxes, int64_t passes, int64_t nch) {
    int S = 1;
    while (S < 8 && 2 * S <= nch && boxes * passes * 2 * S <= (int64_t)device_shape().sms) S *= 2;
    return S;
}

// or over the grid's z without clusters, any count up to 16 while the grid fits the SMs,
// each split's partial tile to a slab of scratch and k_stream_ksum adding the slabs: taken
// where it leaves each CTA fewer chunks than the cluster split (3584 x 18944: 28 boxes x 5
// splits, 8 chunks a CTA, against clusters of 4 and 10; five CTAs of a cluster would not
// pack into the GPCs).  1: the cluster split.
int q6_stream_gsplits(int64_t boxes, int64_t passes, int64_t nch) {
    const int forced = g_small_ksplit.load();  // the test switch: 1 never, n > 1 n splits
    if (forced > 0) return (int)std::min<int64_t>(forced, nch);
    const int64_t sms = device_shape().sms, S = q6_stream_splits(boxes, passes, nch);
    int zg = 1;
    for (int z = 2; z <= 16 && z <= nch && boxes * passes * z <= sms; ++z)
        if ((nch + z - 1) / z < (nch + zg - 1) / zg) zg = z;
    return (nch + zg - 1) / zg < (nch + S - 1) / S ? zg : 1;
}

template <bool DOTS>
int launch_q6_stream_t(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                       int32_t* dots, cudaStream_t s, const char* fn) {
    const int64_t nsb = nb / 8, nch = nsb / 2, boxes = (N + 127) / 128, passes = (M + 7) / 8;
    const int S = q6_stream_splits(boxes, passes, nch);
    const int zg = DOTS || (g_small_ksplit.load() == 0 && N * nsb * Q6_K_BYTES < EAGER_SPLIT_MIN_BYTES &&
                            !stream_captured(s))
                       ? 1
                       : q6_stream_gsplits(boxes, passes, nch);
    static SmemAttr attr, attr_g;
    const int e = zg > 1 ? ensure_smem((const void*)k_mmq_q6_stream<false, true>, Q6S_SMEM, attr_g)
                         : ensure_smem((const void*)k_mmq_q6_stream<DOTS>, Q6S_SMEM, attr);
    if (e != MMQ_OK) {
        report(fn, e, "shared-memory request refused");
        return e;
    }
    CUtensorMap tw, tx, txl;
    if (!make_byte_map(&tw, w8, (uint64_t)nsb * 8 * Q6_K_BYTES, (uint64_t)(N / 8), Q6S_LB, Q6S_LINES, 8) ||
        !make_act_maps(&tx, &txl, x8, M, nb, Q6S_XROW)) {
        report(fn, MMQ_ERR_CUDA, "tensor map encoding failed");
        return MMQ_ERR_CUDA;
    }
    // one chunk's transfer at this CTA's share of about 6 TB/s (bytes / (bytes per ns));
    // at most 2 us (a bounded wait)
    const int64_t ctas = std::min<int64_t>(boxes * passes * std::max(S, zg), device_shape().sms);
    const unsigned stagger = (unsigned)std::min<int64_t>(2000, (int64_t)(Q6S_WBYTES + 8 * Q6S_XROW) * ctas / 6000);
    SplitScratch ss;
    return launch_stream_split(
        zg, M, N, out, s, fn,
        [&](float* o, long long pstride, unsigned gz) {
            ProfScope ps("k_mmq_q6_stream", s);
            const dim3 blk(Q6S_THREADS);
            if (gz > 1) {
                const int st = pdl_status(launch_pdl(k_mmq_q6_stream<false, true>,
                                                     dim3((unsigned)boxes, (unsigned)passes, gz), blk,
                                                     (size_t)Q6S_SMEM, s, tw, tx, txl, (int)M, (int)N, nb, stagger, o,
                                                     pstride, dots),
                                          fn);
                return st == MMQ_OK ? split_scratch_bind(ss, s, fn) : st;
            }
            return pdl_status(launch_pdl_zcluster(k_mmq_q6_stream<DOTS>, dim3((unsigned)boxes, (unsigned)passes,
                                                                                (unsigned)S),
                                                  blk, (size_t)Q6S_SMEM, s, (unsigned)S, tw, tx, txl, (int)M, (int)N,
                                                  nb, stagger, o, pstride, dots),
                              fn);
        },
        &ss);
}

int launch_q6_stream(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out, int32_t* dots,
                     cudaStream_t s, const char* fn) {
    return dots ? launch_q6_stream_t<true>(x8, w8, M, N, nb, out, dots, s, fn)
                : launch_q6_stream_t<false>(x8, w8, M, N, nb, out, dots, s, fn);
}

template <int FMT>
int launch_i8_stream(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                     int32_t* dots, cudaStream_t s, const char* fn) {
    if constexpr (is_kquant(FMT))
        return launch_kq_stream<FMT>(x8, w8, M, N, nb, out, dots, s, fn);
    else
        return launch_i8_stream_q8_0(x8, w8, M, N, nb, out, dots, s, fn);
}

}  // namespace

double q6_stream_cost_us(int64_t M, int64_t N, int64_t K) {
    const int nb = (int)(K / QK);
    if (K % QK_K != 0 || !q6_stream_fits(N, nb)) return -1.0;
    const int64_t nch = nb / 16, boxes = (N + 127) / 128, passes = (M + 7) / 8, sms = device_shape().sms;
    const int64_t zg = q6_stream_gsplits(boxes, passes, nch);
    const int64_t S = zg > 1 ? zg : q6_stream_splits(boxes, passes, nch);
    const int64_t waves = (boxes * passes * S + sms - 1) / sms;
    return (double)(waves * ((nch + S - 1) / S)) * 1.9 + 3.5;
}

// The expert-grouped contraction on the dp4a weight stream (tiles of at most mt = 1, 2 or 4
// rows of one expert, from the grouping kernels): for experts with few rows, where a
// 128-row tensor-core tile would be almost empty and the expanded path would expand every
// such expert's weights.  false from small_grouped_fits: not for this shape.
bool small_grouped_fits(int fmt, int64_t K, int mt) {
    const int nb = (int)(K / QK);
    return nb % 8 == 0 && ds_smem_bytes(fmt, mt <= 1 ? 1 : mt <= 2 ? 2 : 4, mt <= 1 && fmt != FMT_Q6_K ? 2 : 4, nb) <=
                              220 * 1024;
}

int small_grouped_launch(int fmt, const void* xq, const void* wq, int64_t R, int64_t E, int64_t N, int64_t K,
                         const int2* tiles, const int* ntiles, int64_t max_tiles, const int* offsets, const int* perm,
                         int mt, float* out, cudaStream_t s, const char* fn) {
    const int nb = (int)(K / QK);
    const long long row_bytes =
        is_superblock(fmt) ? (long long)(nb / 8) * kq_bytes(fmt) : (long long)nb * Q8_0_BYTES;
    const DsGroup g{tiles, ntiles, offsets, perm, (long long)N * row_bytes, (long long)E * N * row_bytes};
    const uint8_t* x8 = static_cast<const uint8_t*>(xq);
    const uint8_t* w8 = static_cast<const uint8_t*>(wq);
    return fmt == FMT_Q8_0   ? launch_dp4a_grouped<FMT_Q8_0>(x8, w8, R, N, nb, mt, out, s, fn, g, max_tiles)
           : fmt == FMT_Q5_K ? launch_dp4a_grouped<FMT_Q5_K>(x8, w8, R, N, nb, mt, out, s, fn, g, max_tiles)
           : fmt == FMT_Q6_K ? launch_dp4a_grouped<FMT_Q6_K>(x8, w8, R, N, nb, mt, out, s, fn, g, max_tiles)
                             : launch_dp4a_grouped<FMT_Q4_K>(x8, w8, R, N, nb, mt, out, s, fn, g, max_tiles);
}

unsigned small_take_error() {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_small_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_small_error, &zero, sizeof(zero));
    }
    return v;
}

std::atomic<int> g_small_route{SMALL_ROUTE_AUTO};

int small_set_route(int route) { return g_small_route.exchange(route); }

// The grid the Q8_0 / Q4_K / Q5_K tensor-core stream takes for M x N x K under stream
// capture (no eager size floor): boxes per CTA and K splits.  Host only.
void small_stream_grid(int fmt, int64_t M, int64_t N, int64_t K, int32_t* boxes, int32_t* splits) {
    const int nb = (int)(K / QK);
    StreamGrid g{1, 1};
    if (fmt == FMT_Q8_0) {
        g = stream_grid((N + 15) / 16, IS_MAX_TPC, (M + 7) / 8, nb / 8, IS_WARPS, INT64_MAX, nullptr);
    } else {
        const bool wide = (N + 31) / 32 >= 2 * (int64_t)device_shape().sms;
        const int boxr = wide ? 32 : 16;
        g = stream_grid((N + boxr - 1) / boxr, ks_max_boxes(boxr), (M + 7) / 8, nb / 8, ks_warps(fmt, boxr), INT64_MAX,
                        nullptr);
    }
    *boxes = (int32_t)g.tpc;
    *splits = g.z;
}
void small_set_ksplit(int splits, int boxes) {
    g_small_kboxes.store(boxes);
    g_small_ksplit.store(splits);
}

int small_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                 int32_t* dots, cudaStream_t s) {
    const int nb = (int)(K / QK);
    if ((M + SMALL_MT - 1) / SMALL_MT > 65535) {
        report(fmt == FMT_Q8_0 ? "mmq_gemm_q8_0" : "mmq_gemm_q4_k", MMQ_ERR_SHAPE,
               "the warp-level path takes M <= 524280");
        return MMQ_ERR_SHAPE;
    }
    const uint8_t* x8 = static_cast<const uint8_t*>(xq);
    const uint8_t* w8 = static_cast<const uint8_t*>(wq);
    const char* sfn = fmt == FMT_Q8_0   ? "mmq_gemm_q8_0 (small-M)"
                      : fmt == FMT_Q5_K ? "mmq_gemm_q5_k (small-M)"
                      : fmt == FMT_Q6_K ? "mmq_gemm_q6_k (small-M)" : "mmq_gemm_q4_k (small-M)";
    if (fmt == FMT_Q6_K) {
        if (nb % 8 != 0) {
            report(sfn, MMQ_ERR_K_MULTIPLE, "Q6_K needs K % 256 == 0");
            return MMQ_ERR_K_MULTIPLE;
        }
        // the tensor-core stream from two rows on (three on a long K through few rows:
        // 3584 x 18944, two rows: 17.6 us on the dp4a stream against 22.3) where its shape
        // rules hold; else the dp4a weight stream, 1, 2 or 4 activation rows per pass (one
        // row per pass when four rows' activations do not fit in shared memory next to the ring)
        const int route = g_small_route.load();
        const bool q6_long_narrow = (N + 15) / 16 <= 2 * (int64_t)device_shape().sms && nb / 8 >= 32;
        if (q6_stream_fits(N, nb) && route != SMALL_ROUTE_DP4A &&
            (route == SMALL_ROUTE_MMA || M >= (q6_long_narrow ? 3 : 2)))
            return launch_q6_stream(x8, w8, M, N, nb, out, dots, s, sfn);
        const int mt = M <= 1 ? 1 : M <= 2 ? 2 : 4;
        if (ds_smem_bytes(fmt, mt, mt == 1 ? 2 : 4, nb) <= 220 * 1024 && (M + mt - 1) / mt <= 65535)
            return launch_dp4a_stream<FMT_Q6_K>(x8, w8, M, N, nb, out, dots, s, sfn);
        if (ds_smem_bytes(fmt, 1, 2, nb) <= 220 * 1024 && M <= 65535)
            return launch_dp4a_stream_s<FMT_Q6_K, 1, 2>(x8, w8, M, N, nb, out, dots, s, sfn);
        report(sfn, MMQ_ERR_SHAPE, "K or M too large for the Q6_K small-M stream (the expanded path takes it)");
        return MMQ_ERR_SHAPE;
    }
    // measured crossovers (GEMM alone, back-to-back graph launches, 7B projections): the dp4a
    // weight stream for one row (Q4_K 18944 x 3584: 8.7 us against 9.9); for two rows of Q5_K
    // (12.9 against 13.9), and of Q4_K when the tensor-core stream would run few 16-row tiles
    // per SM through a long K (3584 x 18944: 11.9 us against 13.1 with its K split); the
    // tensor-core streams otherwise (Q4_K 4 x 18944 x 3584: 10.1 us against 17.8; on 3584 x
    // 18944 Q8_0 two rows 17.0 against 18.5, Q5_K four rows 16.9 against 18.6)
    const int route = g_small_route.load();
    const bool long_narrow = (N + 15) / 16 <= 2 * (int64_t)device_shape().sms && nb / 8 >= 32;
    const int64_t auto_max = M <= 1                                                         ? 1
                             : (fmt == FMT_Q5_K || (long_narrow && fmt == FMT_Q4_K)) && M <= 2 ? 2
                                                                                             : 0;
    const int64_t dp4a_max_m = route == SMALL_ROUTE_DP4A ? 4 : route == SMALL_ROUTE_MMA ? 0 : auto_max;
    if (nb % 8 == 0 && M <= dp4a_max_m && ds_smem_bytes(fmt, M <= 1 ? 1 : M <= 2 ? 2 : 4, 4, nb) <= 220 * 1024)
        return fmt == FMT_Q8_0   ? launch_dp4a_stream<FMT_Q8_0>(x8, w8, M, N, nb, out, dots, s, sfn)
               : fmt == FMT_Q5_K ? launch_dp4a_stream<FMT_Q5_K>(x8, w8, M, N, nb, out, dots, s, sfn)
                                 : launch_dp4a_stream<FMT_Q4_K>(x8, w8, M, N, nb, out, dots, s, sfn);
    if (nb % 8 == 0)
        return fmt == FMT_Q8_0   ? launch_i8_stream<FMT_Q8_0>(x8, w8, M, N, nb, out, dots, s, sfn)
               : fmt == FMT_Q5_K ? launch_i8_stream<FMT_Q5_K>(x8, w8, M, N, nb, out, dots, s, sfn)
                                 : launch_i8_stream<FMT_Q4_K>(x8, w8, M, N, nb, out, dots, s, sfn);
    if (fmt == FMT_Q5_K) {  // K-quants come in whole super-blocks: nb % 8 == 0 always
        report(sfn, MMQ_ERR_K_MULTIPLE, "Q5_K needs K % 256 == 0");
        return MMQ_ERR_K_MULTIPLE;
    }
    if (nb % 2 == 0) {
        dim3 g2((unsigned)((N + 15) / 16), (unsigned)((M + 7) / 8));
        ProfScope ps("k_mmq_small_mma", s);
        if (fmt == FMT_Q8_0)
            k_mmq_small_mma<FMT_Q8_0><<<g2, MMA_WARPS * 32, 0, s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
        else
            k_mmq_small_mma<FMT_Q4_K><<<g2, MMA_WARPS * 32, 0, s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
        return launch_status(fmt == FMT_Q8_0 ? "mmq_gemm_q8_0 (small-M)" : "mmq_gemm_q4_k (small-M)");
    }
    dim3 grid((unsigned)((N + SMALL_WARPS - 1) / SMALL_WARPS), (unsigned)((M + SMALL_MT - 1) / SMALL_MT));
    ProfScope ps("k_mmq_small", s);
    if (fmt == FMT_Q8_0)
        k_mmq_small<FMT_Q8_0><<<grid, SMALL_WARPS * 32, 0, s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
    else
        k_mmq_small<FMT_Q4_K><<<grid, SMALL_WARPS * 32, 0, s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
    return launch_status(fmt == FMT_Q8_0 ? "mmq_gemm_q8_0 (small-M)" : "mmq_gemm_q4_k (small-M)");
}

}  // namespace mmq
