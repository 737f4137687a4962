// MMQ for few activation rows: the decode-like regime, bound by the weight bytes read
// from HBM ("When Does a Kernel Win Surface?", sec. "A bottleneck taxonomy",
// bandwidth-roofline decode).  Kernels, chosen by small_launch at the end of the file:
//   k_mmq_dp4a_stream  one row (two for Q5_K and long K, up to four in a few cases, see
//                      small_launch): per-warp weight streams, dp4a;
//   k_mmq_i8_stream,   up to eight rows per pass on the tensor cores through mma.sync (Q8_0
//   k_mmq_kq_stream    on s8, the K-quants on f16), per-warp rings of 2-D tensor copies;
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

// S: slots per warp; 4 CTAs per SM with 2 slots, 2 CTAs per SM with 4 (64 copies in flight per SM)
template <int FMT, int MT, int S>
__global__ void __launch_bounds__(DS_WARPS * 32, S == 2 ? 4 : 2)
k_mmq_dp4a_stream(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ wq, int M, int N, int nb,
                  float* __restrict__ out, int32_t* __restrict__ dots) {
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
    const int m0 = blockIdx.y * MT;
    const int ntok = min(MT, M - m0);
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
            const long long a = n * row_bytes + (long long)u0 * UB, end = (long long)N * row_bytes;
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
        ptx::bulk_load(ptx::smem_u32(ring + (q % S) * DS_SLOT), wq + n * row_bytes + (long long)u0 * UB,
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
            const uint32_t* src = reinterpret_cast<const uint32_t*>(xq + ((long long)(m0 + t) * nb + b) * Q8_1_BYTES);
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
                    const int bs = (int)((n * row_bytes + (long long)u0 * UB) & 15) + sl * Q6_K_BYTES;
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
                if (lane == 0 && t < ntok) out[(long long)(m0 + t) * N + n] = v;
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

template <int FMT, int MT, int S>
int launch_dp4a_stream_s(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                         int32_t* dots, cudaStream_t s, const char* fn) {
    const int smem = ds_smem_bytes(FMT, MT, S, nb);
    static SmemAttr attr;
    if (smem > 48 * 1024) {
        const int e = ensure_smem((const void*)k_mmq_dp4a_stream<FMT, MT, S>, smem, attr);
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
    const int64_t rpw = (N + max_warps - 1) / max_warps;
    const int64_t ctas = (N + DS_WARPS * rpw - 1) / (DS_WARPS * rpw);
    dim3 grid((unsigned)ctas, (unsigned)((M + MT - 1) / MT));
    {
        ProfScope ps("k_mmq_dp4a_stream", s);
        return pdl_status(launch_pdl(k_mmq_dp4a_stream<FMT, MT, S>, grid, dim3(DS_WARPS * 32), (size_t)smem, s, x8, w8,
                                     (int)M, (int)N, nb, out, dots),
                          fn);
    }
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

template <bool DOTS>
__global__ void __launch_bounds__(IS_WARPS * 32, 2)
k_mmq_i8_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmXl, int M, int N,
                int nb, int tpc, float* __restrict__ out, int32_t* __restrict__ dots) {
    constexpr int S = I8_SLOTS, SA = I8_ASLOTS, SLOT = I8_SLOT, RB = 8 * Q8_0_BYTES, WB = I8_WARP_BYTES;
    extern __shared__ __align__(128) uint8_t is_smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    uint8_t* ring = is_smem + warp * WB;  // S weight slots, then SA activation slots
    uint8_t* aring = ring + S * SLOT;
    const uint32_t bar0 = ptx::smem_u32(is_smem + IS_WARPS * WB) + 8 * (S + SA) * warp;
    const uint32_t abar0 = bar0 + 8 * S;
    const int ntiles = (N + 15) / 16;
    const int t0 = blockIdx.x * tpc, nt = min(tpc, ntiles - t0);
    const int npieces = nb / 8;  // groups of 8 blocks
    const int my = warp < npieces ? (npieces - 1 - warp) / IS_WARPS + 1 : 0;  // this warp's pieces per tile
    const int total = nt * my;
    const int m0 = blockIdx.y * 8;
    const bool h0ok = m0 + 2 * q < M, h1ok = m0 + 2 * q + 1 < M;  // the D fragment's tokens 2q, 2q + 1

    IsSchedule next{0, 0};
    auto issue = [&](int i) {  // lane 0: the copy of this warp's weight piece i into slot i % S
        const uint32_t bar = bar0 + 8 * (i % S);
        ptx::mbar_arrive_expect_tx(bar, SLOT);  // the whole box, zero-filled rows included
        ptx::tma_load_2d(ptx::smem_u32(ring + (i % S) * SLOT), &tmW, bar, (warp + next.k * IS_WARPS) * (RB / 8),
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
                         (warp + k * IS_WARPS) * (IS_XROW / 8), m0);
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
        const int b0 = 8 * (warp + k * IS_WARPS);  // first block of the piece
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

template <int FMT, int BOXR, bool DOTS>
__global__ void __launch_bounds__(ks_warps(FMT, BOXR) * 32, 2)
k_mmq_kq_stream(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const __grid_constant__ CUtensorMap tmXl, int M, int N,
                int nb, int tpc, float* __restrict__ out, int32_t* __restrict__ dots) {
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
    const int npieces = nb / 8;  // super-blocks
    const int my = warp < npieces ? (npieces - 1 - warp) / W + 1 : 0;  // this warp's pieces per box
    const int total = nt * my;
    const int m0 = blockIdx.y * 8;
    const bool h0ok = m0 + 2 * q < M, h1ok = m0 + 2 * q + 1 < M;  // the D fragment's tokens 2q, 2q + 1

    IsSchedule next{0, 0};
    auto issue = [&](int i) {  // lane 0: the copy of this warp's weight piece i into slot i % S
        const uint32_t bar = bar0 + 8 * (i % S);
        ptx::mbar_arrive_expect_tx(bar, SLOT);  // the whole box, zero-filled rows included
        ptx::tma_load_2d(ptx::smem_u32(ring + (i % S) * SLOT), &tmW, bar, (warp + next.k * W) * (RB / 8),
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
                         (warp + k * W) * (IS_XROW / 8), m0);
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
        const int b0 = 8 * (warp + k * W);  // first block of the piece
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

// the activation maps of the streams: 8-row boxes for the full passes, and for the last pass
// a box of its own rows (M - 8 (passes - 1)); copying rows past M as the copy engine's
// zero fill was measured to slow a one-row pass down by a third
inline bool make_act_maps(CUtensorMap* tx, CUtensorMap* txl, const uint8_t* x8, int64_t M, int nb) {
    const uint32_t last = (uint32_t)(M - 8 * ((M - 1) / 8));
    return make_byte_map(tx, x8, (uint64_t)nb * Q8_1_BYTES, (uint64_t)M, IS_XROW, 8, 8) &&
           make_byte_map(txl, x8, (uint64_t)nb * Q8_1_BYTES, (uint64_t)M, IS_XROW, last, 8);
}

// boxes per CTA: the fewest (at most max_boxes) that keep the grid within the two CTAs per
// SM that are resident at once (no second, partial wave)
inline int64_t stream_tpc(int64_t nboxes, int max_boxes) {
    const int64_t per_wave = 2 * (int64_t)device_shape().sms;
    const int64_t tpc = (nboxes + per_wave - 1) / per_wave;
    return tpc < 1 ? 1 : (tpc > max_boxes ? max_boxes : tpc);
}

int launch_i8_stream_q8_0(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                          int32_t* dots, cudaStream_t s, const char* fn) {
    const int64_t ntiles = (N + 15) / 16;
    const int64_t tpc = stream_tpc(ntiles, IS_MAX_TPC);
    static SmemAttr attr, attr_d;
    const int e = dots ? ensure_smem((const void*)k_mmq_i8_stream<true>, I8_SMEM, attr_d)
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
    dim3 grid((unsigned)((ntiles + tpc - 1) / tpc), (unsigned)((M + 7) / 8));
    ProfScope ps("k_mmq_i8_stream", s);
    return pdl_status(dots ? launch_pdl(k_mmq_i8_stream<true>, grid, dim3(IS_WARPS * 32), (size_t)I8_SMEM, s, tw, tx, txl,
                                        (int)M, (int)N, nb, (int)tpc, out, dots)
                           : launch_pdl(k_mmq_i8_stream<false>, grid, dim3(IS_WARPS * 32), (size_t)I8_SMEM, s, tw, tx, txl,
                                        (int)M, (int)N, nb, (int)tpc, out, dots),
                      fn);
}

template <int FMT, int BOXR>
int launch_kq_stream_b(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out,
                       int32_t* dots, cudaStream_t s, const char* fn) {
    const int64_t nboxes = (N + BOXR - 1) / BOXR;
    const int64_t tpc = stream_tpc(nboxes, ks_max_boxes(BOXR));
    constexpr int smem = ks_smem_bytes(FMT, BOXR);
    static SmemAttr attr, attr_d;
    const int e = dots ? ensure_smem((const void*)k_mmq_kq_stream<FMT, BOXR, true>, smem, attr_d)
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
    dim3 grid((unsigned)((nboxes + tpc - 1) / tpc), (unsigned)((M + 7) / 8));
    const dim3 block(ks_warps(FMT, BOXR) * 32);
    ProfScope ps("k_mmq_kq_stream", s);
    return pdl_status(dots ? launch_pdl(k_mmq_kq_stream<FMT, BOXR, true>, grid, block, (size_t)smem, s, tw, tx, txl, (int)M,
                                        (int)N, nb, (int)tpc, out, dots)
                           : launch_pdl(k_mmq_kq_stream<FMT, BOXR, false>, grid, block, (size_t)smem, s, tw, tx, txl,
                                        (int)M, (int)N, nb, (int)tpc, out, dots),
                      fn);
}

// 32-row boxes when there are at least two of them per SM, else 16-row boxes
template <int FMT>
int launch_kq_stream(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out, int32_t* dots,
                     cudaStream_t s, const char* fn) {
    if ((N + 31) / 32 >= 2 * (int64_t)device_shape().sms)
        return launch_kq_stream_b<FMT, 32>(x8, w8, M, N, nb, out, dots, s, fn);
    return launch_kq_stream_b<FMT, 16>(x8, w8, M, N, nb, out, dots, s, fn);
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
        // the dp4a weight stream, 1, 2 or 4 activation rows per pass (one row per pass when
        // four rows' activations do not fit in shared memory next to the ring)
        if (nb % 8 != 0) {
            report(sfn, MMQ_ERR_K_MULTIPLE, "Q6_K needs K % 256 == 0");
            return MMQ_ERR_K_MULTIPLE;
        }
        const int mt = M <= 1 ? 1 : M <= 2 ? 2 : 4;
        if (ds_smem_bytes(fmt, mt, mt == 1 ? 2 : 4, nb) <= 220 * 1024 && (M + mt - 1) / mt <= 65535)
            return launch_dp4a_stream<FMT_Q6_K>(x8, w8, M, N, nb, out, dots, s, sfn);
        if (ds_smem_bytes(fmt, 1, 2, nb) <= 220 * 1024 && M <= 65535)
            return launch_dp4a_stream_s<FMT_Q6_K, 1, 2>(x8, w8, M, N, nb, out, dots, s, sfn);
        report(sfn, MMQ_ERR_SHAPE, "K or M too large for the Q6_K small-M stream (the expanded path takes it)");
        return MMQ_ERR_SHAPE;
    }
    // measured crossovers (GEMM alone, back-to-back graph launches, 7B projections): the dp4a
    // weight stream for one row (Q4_K 18944 x 3584: 8.7 us against 9.9); for two rows when
    // the tensor-core stream would run one 16-row tile per CTA through a long K (3584 x
    // 18944: 12.0 us against 16.1) or for Q5_K (12.9 against 13.9); for three or four rows
    // only Q5_K on such a long K (18.7 against 20.4); the tensor-core streams otherwise (Q4_K
    // 4 x 18944 x 3584: 10.1 us against 17.8)
    const int route = g_small_route.load();
    const bool long_narrow = (N + 15) / 16 <= 2 * (int64_t)device_shape().sms && nb / 8 >= 32;
    const int64_t auto_max = M <= 1                                  ? 1
                             : (fmt == FMT_Q5_K || long_narrow) && M <= 2 ? 2
                             : fmt == FMT_Q5_K && long_narrow         ? 4
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
