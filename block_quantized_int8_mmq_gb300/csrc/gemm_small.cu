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
//
// For K a multiple of 64 the contraction runs on the tensor cores instead
// (k_mmq_small_mma): mma.sync m16n8k16 with 16 weight rows as the M side and up to 8
// tokens as N, codes converted to exact fp16 in registers.  dp4a would need the whole
// dp4a rate of an SM to keep pace with HBM at 8 tokens; the fp16 mma has 4x that.
// Within one 32-value block the order of k does not change the dot product, so both
// operands use the same permutation of k: thread (g = lane/4, q = lane%4) takes the 8
// consecutive values 8q..8q+7 of the block, i.e. 8 contiguous bytes of a row (Q4_K: one
// 8-byte load gives the low nibbles of sub-block 2c and the high nibbles of 2c+1).
// The 16 warps of a CTA share one 16-row tile and split K; each warp issues every load
// of a batch of chunks (codes, scale headers, activation codes and scales) before any
// math, so the DRAM latency is paid once per batch; the warps reduce through shared
// memory at the end.
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

// ---------------------------------------------------------------- staged variant
// The 16 weight rows of a CTA, and the (at most 8) activation rows, are copied into
// shared memory piece by piece (one bulk copy per row per piece: 2176 B of Q8_0 or
// 2304 B of Q4_K weights), so the whole tile is requested from HBM
// at once and its latency is paid once per piece; the math then reads shared memory.
// Needs K % 256 == 0 (whole 16-byte aligned pieces of both formats).

__device__ unsigned int g_small_error;

constexpr int ST_WARPS = 16;
__host__ __device__ constexpr int st_piece_blocks(int fmt) {  // 32-blocks of K per piece
    return fmt == FMT_Q8_0 ? 64 : 128;
}
constexpr uint64_t ST_WAIT_LIMIT_NS = 2000000000ull;

__host__ __device__ constexpr int st_piece_bytes(int fmt) {
    return fmt == FMT_Q8_0 ? st_piece_blocks(fmt) * Q8_0_BYTES : st_piece_blocks(fmt) / 8 * Q4_K_BYTES;
}

// bytes of activation row data per token per piece in shared memory (padded by 16 B
// so that the 8 token rows start in different banks)
__host__ __device__ constexpr int st_act_stride(int fmt) { return st_piece_blocks(fmt) * Q8_1_BYTES + 16; }
__host__ __device__ constexpr int st_smem_bytes(int fmt) {
    return 16 * st_piece_bytes(fmt) + 8 * st_act_stride(fmt) + ST_WARPS * 16 * 8 * 4 + 16;
}

template <int FMT>
__global__ void __launch_bounds__(ST_WARPS * 32, 2)
k_mmq_small_staged(const uint8_t* __restrict__ xq, const uint8_t* __restrict__ wq, int M, int N, int nb,
                   float* __restrict__ out, int32_t* __restrict__ dots) {
    constexpr int PB = st_piece_bytes(FMT);
    constexpr int PBLK = st_piece_blocks(FMT);
    constexpr int AS = st_act_stride(FMT);
    extern __shared__ __align__(128) uint8_t st_smem[];
    uint8_t* tile = st_smem;                                   // [16 rows][PB]
    uint8_t* act = st_smem + 16 * PB;                          // [8 tokens][AS]
    float(*red)[16][8] = reinterpret_cast<float(*)[16][8]>(act + 8 * AS);
    const uint32_t bar = ptx::smem_u32(act + 8 * AS + ST_WARPS * 16 * 8 * 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int n0 = blockIdx.x * 16, m0 = blockIdx.y * 8;
    const int nrows = min(16, N - n0), ntok = min(8, M - m0);
    const int t0 = 2 * q, t1 = t0 + 1;                         // D-fragment tokens (local)
    const long long row_bytes = FMT == FMT_Q8_0 ? (long long)nb * Q8_0_BYTES : (long long)(nb >> 3) * Q4_K_BYTES;
    const long long xrow_bytes = (long long)nb * Q8_1_BYTES;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    bool ok = true;
    const int npieces = (nb + PBLK - 1) / PBLK;
    for (int p = 0; p < npieces && ok; ++p) {
        const int kb0 = p * PBLK, pb = min(PBLK, nb - kb0);
        const uint32_t bytes = FMT == FMT_Q8_0 ? (uint32_t)pb * Q8_0_BYTES : (uint32_t)(pb >> 3) * Q4_K_BYTES;
        const long long off = FMT == FMT_Q8_0 ? (long long)kb0 * Q8_0_BYTES : (long long)(kb0 >> 3) * Q4_K_BYTES;
        const uint32_t abytes = (uint32_t)pb * Q8_1_BYTES;
        if (threadIdx.x == 0) {
            ptx::mbar_arrive_expect_tx(bar, bytes * (uint32_t)nrows + abytes * (uint32_t)ntok);
            for (int r = 0; r < nrows; ++r)
                ptx::bulk_load(ptx::smem_u32(tile + r * PB), wq + (long long)(n0 + r) * row_bytes + off, bytes, bar);
            for (int t = 0; t < ntok; ++t)
                ptx::bulk_load(ptx::smem_u32(act + t * AS), xq + (long long)(m0 + t) * xrow_bytes + (long long)kb0 * Q8_1_BYTES,
                               abytes, bar);
        }
        if (!ptx::mbar_try_wait(bar, p & 1)) {
            const uint64_t t_start = ptx::globaltimer_ns();
            while (!ptx::mbar_try_wait(bar, p & 1)) {
                if (ptx::globaltimer_ns() - t_start > ST_WAIT_LIMIT_NS) {
                    atomicOr(&g_small_error, ERR_TIMEOUT);
                    ok = false;
                    break;
                }
            }
        }
        if (!ok) break;
        const int rg0 = min(g, nrows - 1), rg1 = min(g + 8, nrows - 1);  // rows past N read row nrows-1 (discarded)
        for (int c = warp; 2 * c < pb; c += ST_WARPS) {
#pragma unroll
            for (int sb = 0; sb < 2; ++sb) {
                const int bl = 2 * c + sb, b = kb0 + bl;     // block within the piece / within the row
                uint32_t a_lo[4], a_hi[4];
                float ws[2], wm[2];
                const int rr[2] = {rg0, rg1};
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint8_t* rowp = tile + rr[i] * PB;
                    if (FMT == FMT_Q4_K) {
                        const uint8_t* sbk = rowp + (bl >> 3) * Q4_K_BYTES;
                        const uint2 wv = *reinterpret_cast<const uint2*>(sbk + 16 + 32 * ((bl >> 1) & 3) + 8 * q);
                        const int shift = 4 * sb;
                        u4x4_h2((wv.x >> shift) & 0x0F0F0F0Fu, a_lo[i], a_lo[i + 2]);
                        u4x4_h2((wv.y >> shift) & 0x0F0F0F0Fu, a_hi[i], a_hi[i + 2]);
                        const uint4 h = *reinterpret_cast<const uint4*>(sbk);
                        int sc, mn;
                        q4_k_scale_min(h.y, h.z, h.w, b & 7, sc, mn);
                        ws[i] = f16_bits_to_f32(h.x) * (float)sc;
                        wm[i] = f16_bits_to_f32(h.x >> 16) * (float)mn;
                    } else {
                        const uint8_t* blk = rowp + bl * Q8_0_BYTES;
                        const int o = 2 + 8 * q + (bl & 1) * 2;     // byte offset of the codes, mod 4
                        const uint32_t* a = reinterpret_cast<const uint32_t*>(blk + 2 + 8 * q - (o & 2));
                        uint32_t w0 = a[0], w1 = a[1];
                        if (o & 2) {
                            const uint32_t w2 = a[2];
                            w0 = __funnelshift_r(w0, w1, 16);
                            w1 = __funnelshift_r(w1, w2, 16);
                        }
                        s8x4_h2(w0, a_lo[i], a_lo[i + 2]);
                        s8x4_h2(w1, a_hi[i], a_hi[i + 2]);
                        ws[i] = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(blk));
                        wm[i] = 0.f;
                    }
                }
                uint32_t xw0 = 0u, xw1 = 0u;
                if (g < ntok) {
                    const uint32_t* xc = reinterpret_cast<const uint32_t*>(act + g * AS + bl * Q8_1_BYTES + 4 + 8 * q);
                    xw0 = xc[0];
                    xw1 = xc[1];
                }
                uint32_t b_lo0, b_lo1, b_hi0, b_hi1;
                s8x4_h2(xw0, b_lo0, b_lo1);
                s8x4_h2(xw1, b_hi0, b_hi1);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma16816(d, a_lo, b_lo0, b_lo1);
                mma16816(d, a_hi, b_hi0, b_hi1);
                if (dots) {
                    const int rw[2] = {n0 + g, n0 + g + 8}, tt[2] = {m0 + t0, m0 + t1};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (rw[e >> 1] < N && tt[e & 1] < M)
                            dots[((long long)tt[e & 1] * N + rw[e >> 1]) * nb + b] = __float2int_rn(d[e]);
                } else {
                    const uint32_t h0 = t0 < ntok ? *reinterpret_cast<const uint32_t*>(act + t0 * AS + bl * Q8_1_BYTES) : 0u;
                    const uint32_t h1 = t1 < ntok ? *reinterpret_cast<const uint32_t*>(act + t1 * AS + bl * Q8_1_BYTES) : 0u;
                    const float xd0 = f16_bits_to_f32(h0), xs0 = f16_bits_to_f32(h0 >> 16);
                    const float xd1 = f16_bits_to_f32(h1), xs1 = f16_bits_to_f32(h1 >> 16);
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
        __syncthreads();  // every warp is done with the tile before the next piece lands
    }
    if (dots || !ok) return;
    red[warp][g][2 * q] = acc[0];
    red[warp][g][2 * q + 1] = acc[1];
    red[warp][g + 8][2 * q] = acc[2];
    red[warp][g + 8][2 * q + 1] = acc[3];
    __syncthreads();
    if (threadIdx.x < 128) {
        const int rr = threadIdx.x >> 3, tt = threadIdx.x & 7;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < ST_WARPS; ++w) v += red[w][rr][tt];
        if (n0 + rr < N && m0 + tt < M) out[(long long)(m0 + tt) * N + n0 + rr] = v;
    }
}

template <int FMT>
int launch_staged(const uint8_t* x8, const uint8_t* w8, int64_t M, int64_t N, int nb, float* out, int32_t* dots,
                  cudaStream_t s) {
    const char* fn = FMT == FMT_Q8_0 ? "mmq_gemm_q8_0 (small-M)" : "mmq_gemm_q4_k (small-M)";
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(k_mmq_small_staged<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             st_smem_bytes(FMT));
        if (e != cudaSuccess) {
            cudaGetLastError();
            report(fn, MMQ_ERR_SMEM, cudaGetErrorString(e));
            return MMQ_ERR_SMEM;
        }
        attr_done = true;
    }
    dim3 grid((unsigned)((N + 15) / 16), (unsigned)((M + 7) / 8));
    {
        ProfScope ps("k_mmq_small_staged", s);
        k_mmq_small_staged<FMT><<<grid, ST_WARPS * 32, st_smem_bytes(FMT), s>>>(x8, w8, (int)M, (int)N, nb, out, dots);
    }
    return launch_status(fn);
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
    if (nb % 8 == 0)
        return fmt == FMT_Q8_0 ? launch_staged<FMT_Q8_0>(x8, w8, M, N, nb, out, dots, s)
                               : launch_staged<FMT_Q4_K>(x8, w8, M, N, nb, out, dots, s);
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
