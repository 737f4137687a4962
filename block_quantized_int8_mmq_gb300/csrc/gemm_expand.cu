// Tensor-core MMQ over codes expanded once per call (sm_103a).
//
// Every int8 code, and every K-quant code (Q4_K: 4 bits, Q5_K: 5 bits) times its 6-bit
// sub-scale, is an exact fp16 value, so the fp16 x fp16 -> f32 MMA over one 32-block
// computes the integer block dot exactly ("When the Product Won't Collapse", sec. "The obstruction": one integer dot
// per constant-scale block).  Because the scale changes at every block, the
// accumulator is read out of TMEM after every block and rescaled in registers (same
// page, sec. "The viable route is per-backend anyway"): out += xd[m,b] * w[n,b] * D_b.
//
// Measured on this GPU, one thread issuing 128 x 128 x 16 MMAs back to back into one
// accumulator gets one every 64 cycles; an item here (one 32-block of a 128 x 128 tile:
// two MMAs for D, one for S, two commits) takes about 750, the chain from issue through
// the commits, the epilogue's TMEM reads and the slot's release, so every tcgen05
// instruction saved per item counts.  Two MMA-issuing warps (even and odd items) each own
// a TMEM slot of 256 columns (D, then the scale products S).
// The codes reach shared memory already in the MMA's layout: one streaming kernel,
// k_expand, converts every code once per call into scratch, its CTAs split between
//
//   activations  q8_1 rows (or f32 rows, quantized on the way) -> per (128-row tile,
//                32-block) an 8 KiB chunk of fp16 codes in the K-major no-swizzle
//                core-matrix order followed by AS_b, the block's K = 16 scale operand
//                (column b % 8 = xd, the other columns 0); per (tile, 256-value group), for
//                K-quants, AM (column c = the f16 block sum s of block c);
//   weights      Q8_0 / Q4_K / Q5_K / Q6_K rows -> per (128-row tile, 32-block) the same
//                chunks (K-quants: q * sc_j; Q6_K: two planes); per (tile, group) WS, the
//                K = 16 operand of the column scales (column c = wd of block c, or d; column
//                8 = -dmin for the min item) and, for K-quants, BMIN (column j = m_j) ("When
//                Does a Kernel Win Surface?", sec. "Kept levers: Vulkan", the Q4_K affine
//                identity);
//
// and k_mmq_tcx copies whole chunks with 1-D bulk copies, issues two K = 16 MMAs per
// block (the exact block dot D) and one K = 16 MMA of AS_b against WS (the scale products
// S = xd (x) w, exact in f32: one nonzero term) per item, and rescales in 16 epilogue
// warps: acc = fma(S, D, acc), one rounding per block.  Rows past M or N are
// zero in the scratch: they add nothing and are never stored.
//
// The price is scratch traffic: 2 bytes written and read back per code.  It pays when
// M is large enough that converting each tile in shared memory, once per output tile
// that uses it, costs more.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"
#include "umma.cuh"

namespace mmq {
namespace {

using namespace umma;

__device__ unsigned long long g_tcx_wait_limit_ns = WAIT_LIMIT_NS;
__device__ unsigned int g_tcx_error;

constexpr int BM = 128;                  // activation rows per tile (TMEM lanes)
constexpr int BN = 128;                  // weight rows per tile (MMA N); the contraction also has 96 (tcx_tile_n)
constexpr int GB = 8;                    // 32-blocks per group (256 values)
constexpr int CHUNK = BM * QK * 2;       // fp16 codes of one block, 128 rows: 8 KiB
constexpr int TILE16 = BM * 16 * 2;      // a K = 16 operand, 128 rows: 4 KiB
constexpr int NSTAGE = 8;                // blocks in flight (one block per stage; Q6_K: 6)
// activation bytes per (tile, block): the fp16 codes, then AS_b, the K = 16 scale operand of
// the block (column b % 8 = xd of the block, the other columns 0)
constexpr int XCHUNK = CHUNK + TILE16;
// weight bytes per (tile, block): one chunk of codes, or for Q6_K two planes whose sum is
// the code times its sub-scale (see expand_weights_q6_k)
__host__ __device__ constexpr int wchunk(int fmt, int bn) { return (fmt == FMT_Q6_K ? 2 : 1) * bn * QK * 2; }
__host__ __device__ constexpr int stage_bytes(int fmt, int bn) { return XCHUNK + wchunk(fmt, bn); }  // activations, then weights
__host__ __device__ constexpr int nstage(int fmt) { return fmt == FMT_Q6_K ? 6 : NSTAGE; }
constexpr int GR = 2;                    // group-data slots
constexpr int NMMA = 2;                  // MMA-issuing warps; warp e issues items e, e + 2, ...
constexpr int DS = NMMA;                 // TMEM slots: slot e (D and S of one item) belongs to issuer e
constexpr int EPI_WARPS = 16;            // warps 0..15: epilogue
constexpr int WARP_LOAD = EPI_WARPS, WARP_MMA0 = EPI_WARPS + 1;
constexpr int THREADS = (WARP_MMA0 + NMMA) * 32;  // 608
constexpr int TMEM_COLS = DS * 2 * BN;            // 512: D at 256e, S at 256e + 128 for either tile width
constexpr int EXP_ROWS = 32;             // rows per expansion CTA (a quarter of a 128-row tile)
constexpr int QCHUNK = EXP_ROWS * QK * 2;     // a chunk's bytes of 32 rows: 2 KiB (whatever the tile's rows)
constexpr int QTILE16 = EXP_ROWS * 16 * 2;    // a K = 16 operand's bytes of 32 rows: 1 KiB
constexpr int EXP_THREADS = 128;

// Group data (scratch and shared memory), per 128-row tile and 256-value group.  Activation
// side: for K-quants AM, the K = 16 operand of the min item (column c = the f16 block sum s
// of block c).  Weight side: for K-quants BMIN (column j = m_j), then WS, the K = 16 operand
// whose column c holds the column scales of item c (Q8_0: wd; K-quants and Q6_K: d; -dmin
// for the min item, column 8).  The scale MMA of block item c multiplies AS_c (only column
// c nonzero: xd) by WS, so S = xd_c (x) w_c exactly; the min item uses a constant AS whose
// column 8 is 1.0.
__host__ __device__ constexpr int xr(int fmt) { return is_kquant(fmt) ? GB + 1 : GB; }
__host__ __device__ constexpr int ga_bytes(int fmt) { return is_kquant(fmt) ? TILE16 : 0; }
__host__ __device__ constexpr int tile16(int rows) { return rows * 16 * 2; }
__host__ __device__ constexpr int gw_bytes(int fmt, int bn) { return (is_kquant(fmt) ? tile16(bn) : 0) + tile16(bn); }
__host__ __device__ constexpr int am_off(int fmt) { return 0; }
__host__ __device__ constexpr int bmin_off(int fmt) { return ga_bytes(fmt); }  // in a group slot: GA, then GW
__host__ __device__ constexpr int ws_off(int fmt, int bn) { return ga_bytes(fmt) + (is_kquant(fmt) ? tile16(bn) : 0); }

__device__ __forceinline__ uint4 pack8(const uint16_t (&v)[8]) {
    return make_uint4(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16), v[4] | ((uint32_t)v[5] << 16),
                      v[6] | ((uint32_t)v[7] << 16));
}

// The device-built row grouping of an expert-grouped call (the grouping kernels of
// grouped.cu): activation tile t holds expert-sorted rows tiles[t].x .. of expert
// tiles[t].y, up to offsets[e + 1] (the expert's end); sorted row m is row perm[m] of the
// caller's activations and output; expert e's weight rows are e * N .. e * N + N - 1 of the
// stacked matrices, in ntpe weight tiles.
struct Grouping {
    const int2* tiles;
    const int* ntiles;
    const int* offsets;
    const int* perm;
    int ntpe;
};

// ---------------------------------------------------------------- expansion kernels
// Piece p (0..511) of a chunk is the 16 bytes of row 8*(p/32) + p%8, values
// 8*((p/8)%4) .. +7 of the block: offset p*16 is that row's core-matrix row, so the
// pieces are written in order (coalesced).

// One CTA per (32-row quarter of a 128-row tile, 256-value group) of the activations, or,
// when it quantizes them (FROM_X) and SPLIT_A, per (quarter, 32-block): the quantization is
// the heavier work, so where the activation tiles are few against the weight tiles it is
// spread over eight times as many CTAs (measured on 512 x 3584 x 3584: 2 blocks per CTA
// 48.5 us per call, 1 block 47.5 us, 8 blocks 50.1 us; on 2048 x 3584 x 18944, where the
// activations are the larger operand, the split cost 1 %).  Rows 32h..32h+31 of
// a tile are row groups 4h..4h+3, i.e. a contiguous 2 KiB of every chunk and 1 KiB of
// every K = 16 tile.  The CTA's q8_1 rows are first gathered into shared memory (row
// stride EXP_SROW): copied from xq, or (FROM_X) quantized here from the f32 rows of x by
// the same per-block arithmetic as k_quantize_q8_1, the q8_1 bytes also written to xq for
// the caller.
constexpr int EXP_SROW = 304;  // 76 words: the 64-bit reads below are conflict-free
// 32-blocks per activation CTA (of a group's 8) and activation CTAs per (quarter, group)
__host__ __device__ constexpr int acts_blocks(bool split) { return split ? 1 : GB; }
__host__ __device__ constexpr int acts_split(bool split) { return GB / acts_blocks(split); }
// the split is taken for the fused quantize when the weight tiles are at least four times
// the activation tiles
__host__ __device__ constexpr bool split_acts(bool from_x, int64_t MT, int64_t NT) { return from_x && NT >= 4 * MT; }

// GROUPED: the quarter's rows are those of activation tile mt of the grouping, read from
// xq through the permutation (tiles past the grouping's count are left alone).
template <int FMT, bool FROM_X, bool SPLIT_A, bool GROUPED>
__device__ __forceinline__ void expand_acts_body(int bx, int g, const float* __restrict__ x,
                                                 const uint8_t* __restrict__ xq_in, uint8_t* __restrict__ xq_out,
                                                 int M, int nb, uint8_t* __restrict__ xa, uint8_t* __restrict__ ga,
                                                 uint8_t* __restrict__ sm, const Grouping& gp) {
    constexpr int ROW = GB * Q8_1_BYTES;  // 288 bytes of one row per group
    constexpr int V = ROW / 16;           // 18
    constexpr int SROW = EXP_SROW;
    static_assert(FROM_X || !SPLIT_A, "the split is for the quantizing expansion");
    constexpr int JB = acts_blocks(SPLIT_A), SPLIT = acts_split(SPLIT_A);
    static_assert(SPLIT == 1 || JB <= 2, "columns of each AM piece");
    static_assert(!GROUPED || !FROM_X, "grouped rows come quantized");
    const int mt = bx / (4 * SPLIT), h = (bx / SPLIT) & 3, j0 = (bx % SPLIT) * JB, ng = nb / GB;
    int m0 = mt * BM + h * EXP_ROWS;
    if constexpr (GROUPED) {
        if (mt >= *gp.ntiles) return;  // uniform over the CTA
        const int2 tl = gp.tiles[mt];
        m0 = tl.x + h * EXP_ROWS;
        M = gp.offsets[tl.y + 1];
    }
    const size_t rowbytes = (size_t)nb * Q8_1_BYTES;
    // shared memory: row r of the quarter, block j0 + jj at r * SROW + jj * 36
    if (FROM_X) {
        // 32 rows x JB blocks, four lanes per block (a pass covers 32 blocks); the loads of
        // BATCH passes are issued before their math
        constexpr int PASSES = EXP_ROWS * JB / (EXP_THREADS / 4);  // 1
        constexpr int BATCH = PASSES < 2 ? PASSES : 2;
        static_assert(PASSES % BATCH == 0, "passes");
        const int part = threadIdx.x & 3;
#pragma unroll
        for (int p0 = 0; p0 < PASSES; p0 += BATCH) {
            float4 va[BATCH], vb[BATCH];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int blk = (p0 + u) * (EXP_THREADS / 4) + (threadIdx.x >> 2);
                const int r = blk / JB, j = j0 + blk % JB, m = m0 + r;
                va[u] = vb[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (m < M) {
                    const float4* src = reinterpret_cast<const float4*>(x + (size_t)m * nb * QK +
                                                                        (size_t)(g * GB + j) * QK + part * 8);
                    va[u] = __ldcs(src);
                    vb[u] = __ldcs(src + 1);
                }
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int blk = (p0 + u) * (EXP_THREADS / 4) + (threadIdx.x >> 2);
                const int r = blk / JB, jj = blk % JB, m = m0 + r;
                const float v[8] = {va[u].x, va[u].y, va[u].z, va[u].w, vb[u].x, vb[u].y, vb[u].z, vb[u].w};
                uint32_t w0, w1, hdr;
                quantize_q8_1_part(v, w0, w1, hdr);
                uint8_t* sb = sm + r * SROW + jj * Q8_1_BYTES;
                if (part == 0) *reinterpret_cast<uint32_t*>(sb) = hdr;
                *reinterpret_cast<uint32_t*>(sb + 4 + 8 * part) = w0;
                *reinterpret_cast<uint32_t*>(sb + 8 + 8 * part) = w1;
                if (m < M) {
                    uint8_t* gb = xq_out + (size_t)m * rowbytes + (size_t)(g * GB + j0 + jj) * Q8_1_BYTES;
                    if (part == 0) *reinterpret_cast<uint32_t*>(gb) = hdr;
                    *reinterpret_cast<uint32_t*>(gb + 4 + 8 * part) = w0;
                    *reinterpret_cast<uint32_t*>(gb + 8 + 8 * part) = w1;
                }
            }
        }
    } else {
        for (int i = threadIdx.x; i < EXP_ROWS * V; i += EXP_THREADS) {
            const int r = i / V, c = i % V;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (m0 + r < M) {
                const int src = GROUPED ? gp.perm[m0 + r] : m0 + r;
                v = __ldg(reinterpret_cast<const uint4*>(xq_in + (size_t)src * rowbytes + (size_t)g * ROW) + c);
            }
            *reinterpret_cast<uint4*>(sm + r * SROW + c * 16) = v;
        }
    }
    __syncthreads();
    uint8_t* dst = xa + ((size_t)mt * nb + (size_t)g * GB + j0) * XCHUNK + h * (CHUNK / 4);
    constexpr int PIECES = CHUNK / 4 / 16;  // 128 16-byte pieces per block per quarter
    for (int i = threadIdx.x; i < JB * PIECES; i += EXP_THREADS) {
        const int jj = i / PIECES, p = i % PIECES;
        const int r = 8 * (p >> 5) + (p & 7), kc = (p >> 3) & 3;  // row within the quarter
        const uint8_t* src = sm + r * SROW + jj * Q8_1_BYTES + 4 + 8 * kc;
        const uint2 lo = i8x4_to_f16x4(*reinterpret_cast<const uint32_t*>(src));
        const uint2 hi = i8x4_to_f16x4(*reinterpret_cast<const uint32_t*>(src + 4));
        *reinterpret_cast<uint4*>(dst + (size_t)jj * XCHUNK + p * 16) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    // AS_j of each block (after its codes): quarter piece u (0..63) = (row 8*(u/16) + u%8,
    // columns 8*((u/8)%2) .. +7); column j holds xd of block j, the others are 0
    uint8_t* adst = xa + ((size_t)mt * nb + (size_t)g * GB + j0) * XCHUNK + CHUNK + h * (TILE16 / 4);
    for (int i = threadIdx.x; i < JB * 64; i += EXP_THREADS) {
        const int jj = i >> 6, u = i & 63, j = j0 + jj;
        const int r = 8 * (u >> 4) + (u & 7), kg = (u >> 3) & 1;
        const uint16_t xd = *reinterpret_cast<const uint16_t*>(sm + r * SROW + jj * Q8_1_BYTES);
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (kg == 0 && e == j) ? xd : (uint16_t)0;
        *reinterpret_cast<uint4*>(adst + (size_t)jj * XCHUNK + u * 16) = pack8(v);
    }
    if (is_kquant(FMT) && threadIdx.x >= 64) {
        // AM (group data): quarter piece u = t - 64, column c = s of block c of the group
        uint8_t* gdst = ga + ((size_t)mt * ng + g) * ga_bytes(FMT) + am_off(FMT) + h * (TILE16 / 4);
        const int u = threadIdx.x - 64;
        const int r = 8 * (u >> 4) + (u & 7), kg = (u >> 3) & 1;
        if (SPLIT == 1) {
            uint16_t v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[e] = kg == 0 ? *reinterpret_cast<const uint16_t*>(sm + r * SROW + e * Q8_1_BYTES + 2) : (uint16_t)0;
            *reinterpret_cast<uint4*>(gdst + u * 16) = pack8(v);
        } else if (kg == 0) {  // column j0 of the piece
            *reinterpret_cast<uint16_t*>(gdst + u * 16 + 2 * j0) = *reinterpret_cast<const uint16_t*>(sm + r * SROW + 2);
        } else if (j0 == 0) {  // columns 8..15 are zero
            *reinterpret_cast<uint4*>(gdst + u * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// One CTA per (32-row quarter of a BNT-row tile, 256-value group) of the weights.  FOLD:
// K-quant codes are q * sc_j (the contraction); without it, the raw nibbles (the block-dot
// test hook).
// GROUPED: weight tile nt is tile nt % ntpe of expert nt / ntpe (experts without rows
// are skipped).
template <int FMT, bool FOLD, int BNT, bool GROUPED>
__device__ __forceinline__ void expand_weights_body(int bx, int g, const uint8_t* __restrict__ wq, int N, int nb,
                                                    uint8_t* __restrict__ xb, uint8_t* __restrict__ gw,
                                                    uint8_t* __restrict__ sm, const Grouping& gp) {
    constexpr int ROW = FMT == FMT_Q8_0 ? GB * Q8_0_BYTES : kq_bytes(FMT);  // 272 / 144 / 176 bytes per row per group
    constexpr int V = ROW / 16;                                             // 17 / 9 / 11
    constexpr int VP = V + 1;                                               // + one zero piece (Q8_0 reads 4 B past)
    constexpr int SROW = FMT == FMT_Q8_0 ? 304 : (FMT == FMT_Q4_K ? 176 : 208);
    static_assert(SROW >= VP * 16 && SROW <= EXP_SROW, "row pad");
    constexpr int QPT = BNT / EXP_ROWS, WCH = wchunk(FMT, BNT);  // quarters per tile, bytes per (tile, block)
    const int nt = bx / QPT, h = bx % QPT, ng = nb / GB;
    // the quarter's first row in wq, and how many of its 32 rows exist
    int w0 = nt * BNT + h * EXP_ROWS, nrows = N - w0;
    if constexpr (GROUPED) {
        const int e = nt / gp.ntpe, local = (nt % gp.ntpe) * BNT + h * EXP_ROWS;
        if (gp.offsets[e] == gp.offsets[e + 1]) return;  // uniform over the CTA
        w0 = e * N + local;
        nrows = N - local;
    }
    const size_t rowbytes = FMT == FMT_Q8_0 ? (size_t)nb * Q8_0_BYTES : (size_t)ng * kq_bytes(FMT);
    {
        // every load of a thread issued before its first store: one memory round trip
        constexpr int TOTAL = EXP_ROWS * VP, NL = (TOTAL + EXP_THREADS - 1) / EXP_THREADS;
        uint4 v[NL];
#pragma unroll
        for (int k = 0; k < NL; ++k) {
            const int i = threadIdx.x + k * EXP_THREADS, r = i / VP, c = i % VP;
            v[k] = make_uint4(0u, 0u, 0u, 0u);
            if (i < TOTAL && c < V && r < nrows)
                v[k] = __ldg(reinterpret_cast<const uint4*>(wq + (size_t)(w0 + r) * rowbytes + (size_t)g * ROW) + c);
        }
#pragma unroll
        for (int k = 0; k < NL; ++k) {
            const int i = threadIdx.x + k * EXP_THREADS;
            if (i < TOTAL) *reinterpret_cast<uint4*>(sm + (i / VP) * SROW + (i % VP) * 16) = v[k];
        }
    }
    __syncthreads();
    uint8_t* dst = xb + ((size_t)nt * nb + (size_t)g * GB) * WCH + h * QCHUNK;
    constexpr int PIECES = QCHUNK / 16;  // 128 16-byte pieces per block per quarter
    for (int i = threadIdx.x; i < GB * PIECES; i += EXP_THREADS) {
        const int j = i / PIECES, p = i % PIECES;
        const int r = 8 * (p >> 5) + (p & 7), kc = (p >> 3) & 3;  // row within the quarter
        const uint8_t* row = sm + r * SROW;
        uint2 lo, hi;
        if (FMT == FMT_Q8_0) {
            // codes of block j start at byte 34j + 2: 2-byte aligned only
            const int off = j * Q8_0_BYTES + 2 + 8 * kc;
            const uint32_t* w = reinterpret_cast<const uint32_t*>(row + (off & ~3));
            const int sh = (off & 3) * 8;
            const uint32_t a0 = w[0], a1 = w[1], a2 = w[2];
            lo = i8x4_to_f16x4(__funnelshift_r(a0, a1, sh));
            hi = i8x4_to_f16x4(__funnelshift_r(a1, a2, sh));
        } else {
            // value 32j + k of the super-block: nibble byte 32*(j/2) + k, low nibble for even j
            // (Q5_K: plus the fifth bit, bit j of high-bit byte k)
            const uint32_t* w = reinterpret_cast<const uint32_t*>(row + kq_qs_off(FMT) + 32 * (j >> 1) + 8 * kc);
            uint32_t a0 = w[0], a1 = w[1];
            if (j & 1) {
                a0 >>= 4;
                a1 >>= 4;
            }
            a0 &= 0x0F0F0F0Fu;
            a1 &= 0x0F0F0F0Fu;
            if (FMT == FMT_Q5_K) {
                const uint32_t* qh = reinterpret_cast<const uint32_t*>(row + 16 + 8 * kc);
                a0 |= ((qh[0] >> j) & 0x01010101u) << 4;
                a1 |= ((qh[1] >> j) & 0x01010101u) << 4;
            }
            int sc = 1, mn;
            if (FOLD) {
                const uint32_t* hw = reinterpret_cast<const uint32_t*>(row);
                q4_k_scale_min(hw[1], hw[2], hw[3], j, sc, mn);
            }
            const __half2 sc2 = __half2half2(__int2half_rn(sc));
            if (FMT == FMT_Q5_K) {
                // codes up to 31: (1024 + q) * sc could exceed the f16 range, so the codes
                // are converted exactly first and then scaled (q * sc <= 1953, exact)
                const __half2 one = __half2half2(__int2half_rn(1));
                const __half2 n1024 = __half2half2(__int2half_rn(-1024));
                const uint2 l = u4x4_scaled_f16x4(a0, one, n1024), h = u4x4_scaled_f16x4(a1, one, n1024);
                lo = make_uint2(h2_bits(__hmul2(bits_h2(l.x), sc2)), h2_bits(__hmul2(bits_h2(l.y), sc2)));
                hi = make_uint2(h2_bits(__hmul2(bits_h2(h.x), sc2)), h2_bits(__hmul2(bits_h2(h.y), sc2)));
            } else {
                const __half2 nsc = __half2half2(__int2half_rn(-1024 * sc));
                lo = u4x4_scaled_f16x4(a0, sc2, nsc);
                hi = u4x4_scaled_f16x4(a1, sc2, nsc);
            }
        }
        *reinterpret_cast<uint4*>(dst + (size_t)j * WCH + p * 16) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    uint8_t* gdst = gw + ((size_t)nt * ng + g) * gw_bytes(FMT, BNT);
    const int t = threadIdx.x;
    // WS (K = 16 operand): quarter piece t (0..63) = (row 8*(t/16) + t%8, columns
    // 8*((t/8)%2) .. +7); column c = the scale of item c for that row
    if (t < 64) {
        const int r = 8 * (t >> 4) + (t & 7), kg = (t >> 3) & 1;
        const uint16_t* hdr = reinterpret_cast<const uint16_t*>(sm + r * SROW);
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = 8 * kg + e;
            if (c >= xr(FMT))
                v[e] = 0;
            else if (FMT == FMT_Q8_0)
                v[e] = *reinterpret_cast<const uint16_t*>(sm + r * SROW + c * Q8_0_BYTES);  // wd
            else
                v[e] = c < GB ? hdr[0] : (uint16_t)(hdr[1] ^ 0x8000u);  // d, or -dmin
        }
        *reinterpret_cast<uint4*>(gdst + ws_off(FMT, BNT) - ga_bytes(FMT) + h * QTILE16 + t * 16) = pack8(v);
    }
    if (is_kquant(FMT) && t >= 64) {
        // BMIN: quarter piece u = t - 64 (0..63) = (row 8*(u/16) + u%8, columns 8*((u/8)%2)
        // .. +7), column j = m_j
        const int u = t - 64;
        const int r = 8 * (u >> 4) + (u & 7), kg = (u >> 3) & 1;
        const uint32_t* hw = reinterpret_cast<const uint32_t*>(sm + r * SROW);
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            int sc, mn;
            q4_k_scale_min(hw[1], hw[2], hw[3], e, sc, mn);
            v[e] = kg == 0 ? __half_as_ushort(__int2half_rn(mn)) : (uint16_t)0;
        }
        *reinterpret_cast<uint4*>(gdst + h * QTILE16 + u * 16) = pack8(v);
    }
}

// Q6_K weights: one CTA per (32-row quarter of a 128-row tile, 256-value group).  A
// weight value is d * sc * (q - 32) with q in 0..63 and an int8 scale sc per 16 values
// ("When Does a Kernel Win Surface?", sec. "Unified dp4a decode cores": 16-element scale
// groups, the q - 32 centring).  The scale changes inside a 32-value block, so it is
// folded into the codes; (q - 32) * sc can reach 4096, past the integers fp16 holds
// exactly, so it is split into two planes that are each exact:
//   P1 = (q - 32) * 2 * (sc >> 1)   (|.| <= 4096, always even)
//   P2 = (q - 32) * (sc & 1)        (|.| <= 32)
// and the contraction takes both planes into the same block dot, which then equals the
// integer sum of u * (q - 32) * sc (|D| < 2^24, exact in f32).  The block's column scale
// is d.  Rows are 2-byte aligned only (210-byte super-blocks): a row's super-block is
// gathered as the 16-byte granules that hold it, and words are read from shared memory
// at the 4-byte boundary below and funnel-shifted into place.
constexpr int Q6_SROW = 240;  // 15 granules: a super-block at any even offset in its first granule
static_assert(Q6_SROW <= EXP_SROW && Q6_SROW >= 16 + Q6_K_BYTES + 14, "row pad");

__device__ __forceinline__ uint2 q6_read8(const uint8_t* p) {  // 8 bytes at an even address
    const uint32_t* w = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(p) & ~(uintptr_t)3);
    const int fs = (int)(reinterpret_cast<uintptr_t>(p) & 2) * 8;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
    return make_uint2(__funnelshift_r(w0, w1, fs), __funnelshift_r(w1, w2, fs));
}

template <int BNT, bool GROUPED>
__device__ __forceinline__ void expand_weights_q6_k(int bx, int g, const uint8_t* __restrict__ wq, int N, int nb,
                                                    uint8_t* __restrict__ xb, uint8_t* __restrict__ gw,
                                                    uint8_t* __restrict__ sm, const Grouping& gp, long long wrows) {
    constexpr int GRAN = Q6_SROW / 16;
    constexpr int QPT = BNT / EXP_ROWS, PLANE = BNT * QK * 2, WCH = wchunk(FMT_Q6_K, BNT);  // two planes
    const int nt = bx / QPT, h = bx % QPT, ng = nb / GB;
    // the quarter's first row in wq, and how many of its 32 rows exist (wq holds wrows rows)
    int w0 = nt * BNT + h * EXP_ROWS, nrows = N - w0;
    if constexpr (GROUPED) {
        const int e = nt / gp.ntpe, local = (nt % gp.ntpe) * BNT + h * EXP_ROWS;
        if (gp.offsets[e] == gp.offsets[e + 1]) return;  // uniform over the CTA
        w0 = e * N + local;
        nrows = N - local;
    }
    const long long rowbytes = (long long)ng * Q6_K_BYTES, end = wrows * rowbytes;
    for (int i = threadIdx.x; i < EXP_ROWS * GRAN; i += EXP_THREADS) {
        const int r = i / GRAN, c = i % GRAN;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < nrows) {
            const long long a = (long long)(w0 + r) * rowbytes + (long long)g * Q6_K_BYTES;
            const long long ga = (a & ~15ll) + 16 * c;
            if (ga < a + Q6_K_BYTES) {
                if (ga + 16 <= end) {
                    v = __ldg(reinterpret_cast<const uint4*>(wq + ga));
                } else {  // the buffer's last bytes, past its last whole granule
                    uint16_t u[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    for (int e = 0; e < 8 && ga + 2 * e < end; ++e)
                        u[e] = __ldg(reinterpret_cast<const uint16_t*>(wq + ga + 2 * e));
                    v = pack8(u);
                }
            }
        }
        *reinterpret_cast<uint4*>(sm + r * Q6_SROW + c * 16) = v;
    }
    __syncthreads();
    auto sblk = [&](int r) -> const uint8_t* {  // super-block of row r of the quarter
        const long long a = (long long)(w0 + r) * rowbytes + (long long)g * Q6_K_BYTES;
        return sm + r * Q6_SROW + (int)(a & 15);
    };
    uint8_t* dst = xb + ((size_t)nt * nb + (size_t)g * GB) * WCH + h * QCHUNK;
    constexpr int PIECES = QCHUNK / 16;  // 128 16-byte pieces per block per quarter
    const __half2 one = __half2half2(__int2half_rn(1));
    const __half2 n1056 = __half2half2(__int2half_rn(-1056));  // 0x6400 | q = 1024 + q; minus 1056 = q - 32
    for (int i = threadIdx.x; i < GB * PIECES; i += EXP_THREADS) {
        const int j = i / PIECES, p = i % PIECES;
        const int r = 8 * (p >> 5) + (p & 7), kc = (p >> 3) & 3;  // row within the quarter, values 8kc .. 8kc + 7
        const uint8_t* sb = sblk(r);
        const int hh = j >> 2, t = j & 3;  // value 32j + 8kc + e = 128 hh + 32 t + (8 kc + e)
        const uint2 lq = q6_read8(sb + 64 * hh + 32 * (t & 1) + 8 * kc);
        const uint2 hq = q6_read8(sb + 128 + 32 * hh + 8 * kc);
        const int sh = 4 * (t >> 1);
        const uint32_t q0 = ((lq.x >> sh) & 0x0F0F0F0Fu) | (((hq.x >> (2 * t)) & 0x03030303u) << 4);
        const uint32_t q1 = ((lq.y >> sh) & 0x0F0F0F0Fu) | (((hq.y >> (2 * t)) & 0x03030303u) << 4);
        const int sc = (int)(int8_t)sb[192 + 2 * j + (kc >> 1)];
        const uint2 c0 = u4x4_scaled_f16x4(q0, one, n1056), c1 = u4x4_scaled_f16x4(q1, one, n1056);  // q - 32
        const __half2 s1 = __half2half2(__int2half_rn(2 * (sc >> 1))), s2 = __half2half2(__int2half_rn(sc & 1));
        const uint4 p1 = make_uint4(h2_bits(__hmul2(bits_h2(c0.x), s1)), h2_bits(__hmul2(bits_h2(c0.y), s1)),
                                    h2_bits(__hmul2(bits_h2(c1.x), s1)), h2_bits(__hmul2(bits_h2(c1.y), s1)));
        const uint4 p2 = make_uint4(h2_bits(__hmul2(bits_h2(c0.x), s2)), h2_bits(__hmul2(bits_h2(c0.y), s2)),
                                    h2_bits(__hmul2(bits_h2(c1.x), s2)), h2_bits(__hmul2(bits_h2(c1.y), s2)));
        *reinterpret_cast<uint4*>(dst + (size_t)j * WCH + p * 16) = p1;
        *reinterpret_cast<uint4*>(dst + (size_t)j * WCH + PLANE + p * 16) = p2;
    }
    // WS (K = 16 operand): quarter piece t (0..63) = (row 8*(t/16) + t%8, columns
    // 8*((t/8)%2) .. +7); columns 0..7 = d of the row's super-block
    const int t = threadIdx.x;
    if (t < 64) {
        const int r = 8 * (t >> 4) + (t & 7), kg = (t >> 3) & 1;
        const uint8_t* sb = sblk(r);
        const uint16_t dd = (uint16_t)(sb[208] | (sb[209] << 8));
        uint16_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = kg == 0 ? dd : (uint16_t)0;
        uint8_t* gdst = gw + ((size_t)nt * ng + g) * gw_bytes(FMT_Q6_K, BNT);
        *reinterpret_cast<uint4*>(gdst + ws_off(FMT_Q6_K, BNT) - ga_bytes(FMT_Q6_K) + h * QTILE16 + t * 16) = pack8(v);
    }
}

// Both expansions in one launch: CTAs 0 .. acts_x - 1 (grid x) expand the activations,
// the rest the weights; grid y = the 256-value group.  The two halves are independent, so
// they run side by side instead of one after the other.
template <int FMT, bool FROM_X, bool FOLD, bool SPLIT_A, int BNT, bool GROUPED = false>
__global__ void __launch_bounds__(EXP_THREADS, 12)
k_expand(const float* __restrict__ x, const uint8_t* __restrict__ xq_in, uint8_t* __restrict__ xq_out,
         const uint8_t* __restrict__ wq, int M, int N, int nb, int acts_x, uint8_t* __restrict__ xa,
         uint8_t* __restrict__ ga, uint8_t* __restrict__ xb, uint8_t* __restrict__ gw, Grouping gp, long long wrows) {
    __shared__ __align__(16) uint8_t sm[EXP_ROWS * EXP_SROW];
    // the contraction's CTAs may be scheduled once every CTA of this grid has started (its
    // set-up then overlaps this grid's last wave); it reads the scratch only after this
    // whole grid has completed and its writes are visible (griddepcontrol.wait)
    ptx::grid_dep_launch_dependents();
    if ((int)blockIdx.x < acts_x) {
        expand_acts_body<FMT, FROM_X, SPLIT_A, GROUPED>(blockIdx.x, blockIdx.y, x, xq_in, xq_out, M, nb, xa, ga, sm,
                                                        gp);
    } else {
        if constexpr (FMT == FMT_Q6_K)  // the sub-scales are always folded (they are inside the block dot)
            expand_weights_q6_k<BNT, GROUPED>(blockIdx.x - acts_x, blockIdx.y, wq, N, nb, xb, gw, sm, gp, wrows);
        else
            expand_weights_body<FMT, FOLD, BNT, GROUPED>(blockIdx.x - acts_x, blockIdx.y, wq, N, nb, xb, gw, sm, gp);
    }
}

// ---------------------------------------------------------------- GEMM kernel
constexpr int BAR_ST_FULL = 0, BAR_ST_EMPTY = BAR_ST_FULL + NSTAGE, BAR_G_FULL = BAR_ST_EMPTY + NSTAGE,
              BAR_G_EMPTY = BAR_G_FULL + GR, BAR_D_FULL = BAR_G_EMPTY + GR, BAR_D_EMPTY = BAR_D_FULL + DS,
              BAR_DRAIN = BAR_D_EMPTY + DS, NBARS = BAR_DRAIN + NMMA;

template <int FMT, int BNT>
struct XLayout {
    static constexpr int stages = 0;
    static constexpr int gslot = (ga_bytes(FMT) + gw_bytes(FMT, BNT) + 1023) & ~1023;
    static constexpr int groups = stages + nstage(FMT) * stage_bytes(FMT, BNT);
    static constexpr int asmin = groups + GR * gslot;  // the min item's constant AS (column 8 = 1.0)
    static constexpr int bars = asmin + TILE16;
    static constexpr int tmem_slot = bars + NBARS * 8;
    static constexpr int total = tmem_slot + 16;
    static constexpr int alloc = total + 1024;  // slack to align the base to 1 KiB
    static_assert(alloc <= 227 * 1024, "shared memory");
};

// Warps 0..15 own 32 rows each (their TMEM lane quarter, warp % 4) and a quarter of the
// tile's columns (32 of a 128 x 128 tile, 24 of a 128 x 96 one); warp 16 is the bulk-copy producer; warps 17 and 18 issue the MMAs
// of the even and odd items, each into its own TMEM slot (D at column 256e, S at 256e +
// 128).  The scale MMA of block item c multiplies AS_c, which arrives with the block's codes
// (only column c nonzero: xd), by the group's WS (column c = the item's column scales), so
// S = xd_c (x) w_c exactly.  An item issues three MMAs and two commits (stage free; D and
// S ready).  Epilogue warp 0 releases the
// group data after each group's last item.  Each epilogue warp reads D and S in two
// loads (16 columns, then the other 16 or 8) and hands the slot back before its last FMAs.  With K split over
// gridDim.z CTAs per tile (small outputs), CTA z takes its share of the groups and writes
// a partial tile.
//
// GROUPED (expert-grouped call): CTA (x, y) takes weight tile x of the expert of
// activation tile y of the grouping (CTAs past its count leave at once): the CTAs of one
// activation tile are consecutive, and so are the tiles of one expert, so both operands
// are reused from L2.  Sorted row m of the tile is stored to output row perm[m]; rows of
// the next expert are not stored.
template <int FMT, bool DOTS, int BNT, bool GROUPED = false>
__global__ void __launch_bounds__(THREADS, 1)
k_mmq_tcx(const uint8_t* __restrict__ xa, const uint8_t* __restrict__ ga, const uint8_t* __restrict__ xb,
          const uint8_t* __restrict__ gw, int M, int N, int nb, float* __restrict__ out, int32_t* __restrict__ dots,
          long long split_stride, Grouping gp) {
    using L = XLayout<FMT, BNT>;
    constexpr bool MIN = is_kquant(FMT) && !DOTS;  // a min item closes every group
    constexpr int IPG = GB + (MIN ? 1 : 0);         // items per group
    constexpr int GA = ga_bytes(FMT), GW = gw_bytes(FMT, BNT), WCH = wchunk(FMT, BNT), STAGE = stage_bytes(FMT, BNT);
    constexpr int EPI_COLS = BNT / (EPI_WARPS / 4);  // columns per epilogue warp: 32 (or 24)
    constexpr int H1 = EPI_COLS - 16;               // the second TMEM load's columns: 16 (or 8)
    static_assert(BNT == 128 || (BNT == 96 && !DOTS), "96-wide tiles for the contraction only");
    static_assert(!GROUPED || !DOTS, "grouped calls are contractions");
    constexpr int NS = nstage(FMT);
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = GROUPED ? blockIdx.y : blockIdx.x, nt = GROUPED ? blockIdx.x : blockIdx.y;
    const int n0 = nt * BNT;
    int m0 = mt * BM, wt = nt;  // first activation row; weight tile
    if constexpr (GROUPED) {
        // the tile list was written before the expansion: read it once that has completed
        ptx::grid_dep_wait();
        if (mt >= *gp.ntiles) return;  // uniform over the CTA: nothing set up yet
        const int2 tl = gp.tiles[mt];
        m0 = tl.x;
        M = gp.offsets[tl.y + 1];
        wt = tl.y * gp.ntpe + nt;
    }
    const int ng = nb / GB;
    // K split z of gridDim.z takes groups g0 .. g1 - 1 and writes its partial tile to
    // out + z * split_stride (one split: the output itself); the indices below (items,
    // stages, groups) count from g0
    const int g0 = (int)((long long)blockIdx.z * ng / gridDim.z), g1 = (int)((long long)(blockIdx.z + 1) * ng / gridDim.z);
    const int ngl = g1 - g0;
    const int nitems = ngl * IPG;
    volatile int* abort = &s_abort;
    unsigned* err = &g_tcx_error;
    const uint64_t limit = g_tcx_wait_limit_ns;
    auto bar = [&](int i) -> uint32_t { return sbase + L::bars + 8 * i; };

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < NSTAGE; ++i) {
            ptx::mbar_init(bar(BAR_ST_FULL + i), 1);
            ptx::mbar_init(bar(BAR_ST_EMPTY + i), 1);
        }
        for (int i = 0; i < GR; ++i) {
            ptx::mbar_init(bar(BAR_G_FULL + i), 1);
            ptx::mbar_init(bar(BAR_G_EMPTY + i), 1);  // epilogue warp 0, once the group's last item is done
        }
        for (int i = 0; i < DS; ++i) {
            ptx::mbar_init(bar(BAR_D_FULL + i), 1);
            ptx::mbar_init(bar(BAR_D_EMPTY + i), EPI_WARPS);
        }
        for (int i = 0; i < NMMA; ++i) ptx::mbar_init(bar(BAR_DRAIN + i), 1);
        ptx::fence_barrier_init();
    }
    // the min item's AS: column 8 = 1.0 in every row (K = 16 no-swizzle core-matrix layout:
    // columns 8..15 of row r are the 16 bytes at (r / 8) * 256 + 128 + (r % 8) * 16)
    for (int i = threadIdx.x; i < TILE16 / 16; i += THREADS) {
        const bool hi = ((i >> 3) & 1) != 0;  // the 16-byte piece holds columns 8..15
        reinterpret_cast<uint4*>(smem + L::asmin)[i] = make_uint4(hi ? 0x3C00u : 0u, 0u, 0u, 0u);
    }
    ptx::fence_proxy_async_smem();
    if (warp == WARP_MMA0) {
        ptx::tmem_alloc(sbase + L::tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::tmem_slot);

    if (warp == WARP_LOAD) {
        // ------------------------------------------------------------ bulk-copy producer
        if (lane == 0) {
            // launched as a programmatic dependent of the expansion: everything above
            // overlapped its tail; the scratch it wrote is read from here on
            ptx::grid_dep_wait();
            int st_issued = 0, g_issued = 0;
            bool ok = true;
            for (int g = 0; g < ngl && ok; ++g) {
                const int gg = g0 + g;  // the group's index in K
                if (!DOTS) {
                    const int gs = g % GR;
                    if (!wait_bar(bar(BAR_G_EMPTY + gs), ((g / GR) & 1) ^ 1, abort, err)) break;
                    const uint32_t dst = sbase + L::groups + gs * L::gslot;
                    ptx::mbar_arrive_expect_tx(bar(BAR_G_FULL + gs), GA + GW);
                    if (GA > 0) ptx::bulk_load(dst, ga + ((size_t)mt * ng + gg) * GA, GA, bar(BAR_G_FULL + gs));
                    ptx::bulk_load(dst + GA, gw + ((size_t)wt * ng + gg) * GW, GW, bar(BAR_G_FULL + gs));
                    g_issued = g + 1;
                }
                for (int j = 0; j < GB; ++j) {
                    const int k = g * GB + j, s = k % NS, kk = gg * GB + j;
                    if (!wait_bar(bar(BAR_ST_EMPTY + s), ((k / NS) & 1) ^ 1, abort, err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sbase + L::stages + s * STAGE;
                    ptx::mbar_arrive_expect_tx(bar(BAR_ST_FULL + s), STAGE);
                    ptx::bulk_load(dst, xa + ((size_t)mt * nb + kk) * XCHUNK, XCHUNK, bar(BAR_ST_FULL + s));
                    ptx::bulk_load(dst + XCHUNK, xb + ((size_t)wt * nb + kk) * WCH, WCH, bar(BAR_ST_FULL + s));
                    st_issued = k + 1;
                }
            }
            // copies of the last stages and groups may still be in flight after an abort
            for (int k = st_issued - NS < 0 ? 0 : st_issued - NS; k < st_issued; ++k)
                drain_bar(bar(BAR_ST_FULL + k % NS), (k / NS) & 1, err);
            for (int g = g_issued - GR < 0 ? 0 : g_issued - GR; g < g_issued; ++g)
                drain_bar(bar(BAR_G_FULL + g % GR), (g / GR) & 1, err);
        }
    } else if (warp >= WARP_MMA0 && warp < WARP_MMA0 + NMMA) {
        // ------------------------------------------------------------ MMA issuers
        // Two issuing threads keep the tensor core busy although each switches between
        // the D and S accumulators of its slot at every item.
        const int e = warp - WARP_MMA0;
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(BM, BNT);
            const uint32_t d = tmem + (uint32_t)(e * 2 * BN), sd = d + BN;
            for (int it = e, n = 0; it < nitems; it += NMMA, ++n) {
                const int g = it / IPG, c = it % IPG, gs = g % GR;
                const bool block = c < GB;
                const int k = g * GB + c, s = k % NS;  // block index = stage sequence number
                const uint32_t gbase = sbase + L::groups + gs * L::gslot;
                // a barrier probe costs ~100 cycles even when the phase is complete: the group
                // barrier is probed at this warp's first item of the group only, and the
                // item's probes are issued together (the slow path waits one by one)
                if (!DOTS && (it - NMMA < g * IPG) && !wait_bar(bar(BAR_G_FULL + gs), (g / GR) & 1, abort, err))
                    break;
                const bool r1 = !block || ptx::mbar_test_wait(bar(BAR_ST_FULL + s), (k / NS) & 1);
                const bool r2 = ptx::mbar_test_wait(bar(BAR_D_EMPTY + e), (n & 1) ^ 1);
                if (!(r1 && r2)) {
                    // (the one wait with the run-time bound: the test setting of 0 makes the first
                    // item's wait for a copy just started give up)
                    if (block && !wait_bar_bounded(bar(BAR_ST_FULL + s), (k / NS) & 1, abort, err, limit)) break;
                    if (!wait_bar(bar(BAR_D_EMPTY + e), (n & 1) ^ 1, abort, err)) break;
                }
                ptx::tc_fence_after();
                const uint32_t a = sbase + L::stages + s * STAGE, b = a + XCHUNK;
                if (block) {
                    ptx::umma_f16(d, sdesc(a, 512), sdesc(b, 512), idesc, 0u);
                    ptx::umma_f16(d, sdesc(a + 256, 512), sdesc(b + 256, 512), idesc, 1u);
                    if (FMT == FMT_Q6_K) {  // the second weight plane into the same block dot
                        ptx::umma_f16(d, sdesc(a, 512), sdesc(b + BNT * QK * 2, 512), idesc, 1u);
                        ptx::umma_f16(d, sdesc(a + 256, 512), sdesc(b + BNT * QK * 2 + 256, 512), idesc, 1u);
                    }
                } else {
                    // min item: AM x BMIN^T = sum_j s_j * m_j
                    ptx::umma_f16(d, sdesc(gbase + am_off(FMT), 256), sdesc(gbase + bmin_off(FMT), 256), idesc, 0u);
                }
                if (!DOTS) {
                    // S = AS x WS^T: AS_c (with the block's codes) or the min item's constant AS
                    const uint32_t as = block ? a + CHUNK : sbase + L::asmin;
                    ptx::umma_f16(sd, sdesc(as, 256), sdesc(gbase + ws_off(FMT, BNT), 256), idesc, 0u);
                }
                // the stage (codes and AS_b) is free once these MMAs are done; the group data
                // is released by the epilogue, which takes the items in order, after the
                // group's last item (a commit per group and issuer costs the tensor core as
                // much as an MMA)
                if (block) ptx::umma_commit(bar(BAR_ST_EMPTY + s));
                ptx::umma_commit(bar(BAR_D_FULL + e));
            }
            ptx::umma_commit(bar(BAR_DRAIN + e));  // arrives once every MMA this thread issued is done
            drain_bar(bar(BAR_DRAIN + e), 0, err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3, cg = warp >> 2;
        const int c0 = cg * EPI_COLS;
        const int mrow = m0 + 32 * q + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        unsigned long long acc[EPI_COLS / 2];
#pragma unroll
        for (int c = 0; c < EPI_COLS / 2; ++c) acc[c] = 0ull;
        for (int it = 0; it < nitems; ++it) {
            const int e = it % DS;
            if (!warp_wait(bar(BAR_D_FULL + e), (it / DS) & 1, abort, err)) break;
            ptx::tc_fence_after();
            if (!DOTS && warp == 0 && lane == 0 && it % IPG == IPG - 1) {
                // every MMA of the group's last item and, since the items are taken in order,
                // of all its earlier ones is done: the group data may be overwritten
                ptx::mbar_arrive(bar(BAR_G_EMPTY + (it / IPG) % GR));
            }
            const uint32_t taddr = lane_base + (uint32_t)(e * 2 * BN);
            if constexpr (DOTS) {
                uint32_t dv[EPI_COLS];
                ptx::tmem_ld_cols(taddr, dv);
                ptx::tmem_ld_wait(dv);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BAR_D_EMPTY + e));
                if (mrow < M) {
#pragma unroll
                    for (int j = 0; j < EPI_COLS; ++j) {
                        const int n = n0 + c0 + j;
                        if (n < N)
                            dots[((long long)mrow * N + n) * nb + g0 * GB + it] = __float2int_rn(__uint_as_float(dv[j]));
                    }
                }
            } else {
                {
                    uint32_t dv[16], sv[16];
                    ptx::tmem_ld_cols(taddr, dv);
                    ptx::tmem_ld_cols(taddr + BN, sv);
                    ptx::tmem_ld_wait(dv);
                    ptx::tmem_ld_wait(sv);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[j] = ptx::fma_f32x2(ptx::f2_bits(__uint_as_float(sv[2 * j]), __uint_as_float(sv[2 * j + 1])),
                                                ptx::f2_bits(__uint_as_float(dv[2 * j]), __uint_as_float(dv[2 * j + 1])),
                                                acc[j]);
                }
                {
                    uint32_t dv[H1], sv[H1];
                    ptx::tmem_ld_cols(taddr + 16, dv);
                    ptx::tmem_ld_cols(taddr + BN + 16, sv);
                    ptx::tmem_ld_wait(dv);
                    ptx::tmem_ld_wait(sv);
                    // the whole item is in registers: hand the TMEM slot back
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(BAR_D_EMPTY + e));
#pragma unroll
                    for (int j = 0; j < H1 / 2; ++j)
                        acc[8 + j] =
                            ptx::fma_f32x2(ptx::f2_bits(__uint_as_float(sv[2 * j]), __uint_as_float(sv[2 * j + 1])),
                                           ptx::f2_bits(__uint_as_float(dv[2 * j]), __uint_as_float(dv[2 * j + 1])),
                                           acc[8 + j]);
                }
            }
        }
        // the partial sums may now be read by a dependent launch once this grid is done
        ptx::grid_dep_launch_dependents();
        if (!DOTS && !*abort && mrow < M) {
            const int orow_i = GROUPED ? gp.perm[mrow] : mrow;
            float* orow = out + blockIdx.z * split_stride + (long long)orow_i * N + n0 + c0;
            const int ncols = N - (n0 + c0);  // columns of this warp's EPI_COLS that exist
            if (ncols >= EPI_COLS && (N & 3) == 0) {
#pragma unroll
                for (int c = 0; c < EPI_COLS / 4; ++c)
                    reinterpret_cast<ulonglong2*>(orow)[c] = make_ulonglong2(acc[2 * c], acc[2 * c + 1]);
            } else {
#pragma unroll
                for (int c = 0; c < EPI_COLS / 2; ++c) {
                    if (2 * c < ncols) orow[2 * c] = __uint_as_float((uint32_t)acc[c]);
                    if (2 * c + 1 < ncols) orow[2 * c + 1] = __uint_as_float((uint32_t)(acc[c] >> 32));
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA0) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// The K splits of one output: element i of out is the sum of the splits' partial tiles in
// the order z = 0, 1, ... (the same order at every call: deterministic).  Launched as a
// programmatic dependent of the contraction.
__global__ void __launch_bounds__(256) k_splitk_sum(const float* __restrict__ part, int splits, long long stride,
                                                    long long n, float* __restrict__ out) {
    ptx::grid_dep_wait();
    const long long n4 = n >> 2;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
        float4 a = __ldcs(reinterpret_cast<const float4*>(part) + i);
        for (int z = 1; z < splits; ++z) {
            const float4 b = __ldcs(reinterpret_cast<const float4*>(part + z * stride) + i);
            a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
        }
        reinterpret_cast<float4*>(out)[i] = a;
    }
    const long long t = (n4 << 2) + blockIdx.x * (long long)blockDim.x + threadIdx.x;
    if (t < n && blockIdx.x * (long long)blockDim.x + threadIdx.x < 4) {
        float a = part[t];
        for (int z = 1; z < splits; ++z) a += part[z * stride + t];
        out[t] = a;
    }
}

// ---------------------------------------------------------------- host side
// Scratch comes from a library-owned stream-ordered pool per device: allocated and
// freed on the call's stream, so calls on different streams never share bytes, and
// kept cached between calls (release threshold = no limit).  Under stream capture the
// same two calls are made on the device's default pool, which the graph turns into
// allocation and free nodes.
std::mutex g_pool_mu;
cudaMemPool_t g_pool[MAX_DEVICES];
bool g_pool_tried[MAX_DEVICES];

cudaMemPool_t scratch_pool(int dev) {
    if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lk(g_pool_mu);
    if (!g_pool_tried[dev]) {
        g_pool_tried[dev] = true;
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) == cudaSuccess) {
            uint64_t thr = ~0ull;
            cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &thr);
            g_pool[dev] = p;
        } else {
            cudaGetLastError();
        }
    }
    return g_pool[dev];
}

// Scratch bytes of one call: expanded activations, activation group data, expanded
// weights, weight group data (each a multiple of 256 bytes), and with K splits their f32
// partial outputs (`splits` slabs of M x N, each padded to 256 bytes).
struct ScratchPlan {
    size_t xa, ga, xb, gw, part;
    int splits;
    long long split_stride;  // floats from one slab to the next
    size_t total() const { return xa + ga + xb + gw + part; }
};
ScratchPlan plan_scratch(int fmt, int64_t M, int64_t N, int64_t K, int bn, bool allow_split = true) {
    const int64_t nb = K / QK, ng = nb / GB;
    const int64_t MT = (M + BM - 1) / BM, NT = (N + bn - 1) / bn;
    const int splits = allow_split ? tcx_splits(fmt, M, N, K) : 1;
    const long long stride = ((long long)(M * N) + 63) & ~63LL;
    return {(size_t)(MT * nb) * XCHUNK,
            (size_t)(MT * ng) * ga_bytes(fmt),
            (size_t)(NT * nb) * wchunk(fmt, bn),
            (size_t)(NT * ng) * gw_bytes(fmt, bn),
            splits > 1 ? (size_t)splits * (size_t)stride * 4 : 0,
            splits,
            stride};
}

// The two launches of the path on scratch `ws` (plan_scratch(FMT, M, N, K, BNT) bytes):
// both expansions, then the contraction, in BNT-wide weight tiles.  x != nullptr: the
// activations come as f32 rows and are quantized by the expansion (q8_1 bytes written to
// xq); else xq is the input.
template <int FMT, bool DOTS, bool FOLD, int BNT>
int launch_on(const float* x, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
              int32_t* dots, uint8_t* ws, const ScratchPlan& sp, cudaStream_t s, const char* fn) {
    const int nb = (int)(K / QK), ng = nb / GB;
    const int64_t MT = (M + BM - 1) / BM, NT = (N + BNT - 1) / BNT;
    static SmemAttr attr;
    const int st_attr = ensure_smem((const void*)k_mmq_tcx<FMT, DOTS, BNT>, XLayout<FMT, BNT>::alloc, attr);
    if (st_attr != MMQ_OK) {
        report(fn, st_attr, "shared-memory request refused");
        return st_attr;
    }
    uint8_t* xa = ws;
    uint8_t* ga = xa + sp.xa;
    uint8_t* xb = ga + sp.ga;
    uint8_t* gw = xb + sp.xb;
    float* part = reinterpret_cast<float*>(gw + sp.gw);
    // the block dots of each split go straight to their own places: only the f32 output
    // needs the partial slabs
    const bool summed = sp.splits > 1 && !DOTS;
    // activation CTAs first: 4 per tile (one per quarter), times the block split when they
    // also quantize
    const bool split = split_acts(x && !DOTS, MT, NT);
    const int64_t acts_x = 4 * MT * acts_split(split);
    const dim3 eg((unsigned)(acts_x + (BNT / EXP_ROWS) * NT), (unsigned)ng);
    {
        ProfScope ps("k_expand", s);
        uint8_t* xq_out = static_cast<uint8_t*>(const_cast<void*>(xq));
        const uint8_t* w8 = static_cast<const uint8_t*>(wq);
        if (x && !DOTS && split)
            k_expand<FMT, true, true, true, BNT><<<eg, EXP_THREADS, 0, s>>>(x, nullptr, xq_out, w8, (int)M, (int)N, nb,
                                                                            (int)acts_x, xa, ga, xb, gw, Grouping{}, N);
        else if (x && !DOTS)
            k_expand<FMT, true, true, false, BNT><<<eg, EXP_THREADS, 0, s>>>(x, nullptr, xq_out, w8, (int)M, (int)N,
                                                                             nb, (int)acts_x, xa, ga, xb, gw, Grouping{},
                                                                             N);
        else
            k_expand<FMT, false, FOLD, false, BNT><<<eg, EXP_THREADS, 0, s>>>(
                nullptr, static_cast<const uint8_t*>(xq), nullptr, w8, (int)M, (int)N, nb, (int)acts_x, xa, ga, xb, gw,
                Grouping{}, N);
    }

    {
        // a programmatic dependent launch: the contraction's CTAs may be scheduled while the
        // expansion drains, their set-up (barriers, TMEM, the constant scale operand) overlapping it
        ProfScope ps("k_mmq_tcx", s);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)MT, (unsigned)NT, (unsigned)sp.splits);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = XLayout<FMT, BNT>::alloc;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e =
            cudaLaunchKernelEx(&cfg, k_mmq_tcx<FMT, DOTS, BNT>, (const uint8_t*)xa, (const uint8_t*)ga, (const uint8_t*)xb,
                               (const uint8_t*)gw, (int)M, (int)N, nb, summed ? part : out, dots,
                               summed ? sp.split_stride : 0LL, Grouping{});
        if (e != cudaSuccess) {
            cudaGetLastError();
            report(fn, MMQ_ERR_LAUNCH, cudaGetErrorString(e));
            return MMQ_ERR_LAUNCH;
        }
    }
    if (summed) {
        ProfScope ps("k_splitk_sum", s);
        const long long n = (long long)M * N;
        cudaLaunchConfig_t cfg = {};
        const long long blocks = ((n >> 2) + 255) / 256;
        const long long cap = 4LL * device_shape().sms;
        cfg.gridDim = dim3((unsigned)(blocks < 1 ? 1 : blocks > cap ? cap : blocks));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, k_splitk_sum, (const float*)part, sp.splits, sp.split_stride, n, out);
        if (e != cudaSuccess) {
            cudaGetLastError();
            report(fn, MMQ_ERR_LAUNCH, cudaGetErrorString(e));
            return MMQ_ERR_LAUNCH;
        }
    }
    return launch_status(fn);
}

// The launches in the tile width tcx_tile_n picks (the block-dot hooks: always 128).
template <int FMT, bool DOTS, bool FOLD>
int launch_bn(int bn, const float* x, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
              int32_t* dots, uint8_t* ws, const ScratchPlan& sp, cudaStream_t s, const char* fn) {
    if constexpr (!DOTS)
        if (bn == 96) return launch_on<FMT, DOTS, FOLD, 96>(x, xq, wq, M, N, K, out, dots, ws, sp, s, fn);
    return launch_on<FMT, DOTS, FOLD, BN>(x, xq, wq, M, N, K, out, dots, ws, sp, s, fn);
}

template <int FMT, bool DOTS, bool FOLD = !DOTS>
int launch_x(const float* x, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
             int32_t* dots, cudaStream_t s, const char* fn) {
    void* ws = nullptr;
    const int bn = DOTS ? BN : tcx_tile_n(FMT, M, N);
    const ScratchPlan sp = plan_scratch(FMT, M, N, K, bn);
    const int st0 = scratch_alloc(sp.total(), s, &ws, fn);
    if (st0 != MMQ_OK) return st0;
    const int st = launch_bn<FMT, DOTS, FOLD>(bn, x, xq, wq, M, N, K, out, dots, static_cast<uint8_t*>(ws), sp, s, fn);
    scratch_free(ws, s);  // stream-ordered: after the kernels above
    return st;
}

// ---------------------------------------------------------------- fixed scratch
// The scratch of mmq_gemm_noalloc: a fixed array in the module's device memory, one per
// device, whose address is looked up once per device.  The expansion kernels write
// every byte the GEMM kernel reads (rows past M or N included), so nothing in it has to
// start at zero and nothing is cleared between calls.
constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)64 << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mu;
uint8_t* g_noalloc_ptr[MAX_DEVICES];

uint8_t* noalloc_scratch(int dev) {
    if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
    }
    return g_noalloc_ptr[dev];
}

}  // namespace

// Stream-ordered scratch: from the library's pool of the current device, or, while `s`
// is being captured, the device's default pool (the graph's own allocation and free
// nodes).  Returns MMQ_OK, MMQ_ERR_CUDA or MMQ_ERR_NOMEM (reported).
int scratch_alloc(size_t bytes, cudaStream_t s, void** p, const char* fn) {
    *p = nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_CUDA, "cudaGetDevice failed");
        return MMQ_ERR_CUDA;
    }
    cudaMemPool_t pool = scratch_pool(dev);
    if (!pool) {
        report(fn, MMQ_ERR_CUDA, "scratch pool creation failed");
        return MMQ_ERR_CUDA;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_CUDA, "cudaStreamIsCapturing failed");
        return MMQ_ERR_CUDA;
    }
    const cudaError_t ae = cs == cudaStreamCaptureStatusNone ? cudaMallocFromPoolAsync(p, bytes, pool, s)
                                                            : cudaMallocAsync(p, bytes, s);
    if (ae != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        report(fn, MMQ_ERR_NOMEM, "scratch allocation failed");
        return MMQ_ERR_NOMEM;
    }
    return MMQ_OK;
}

void scratch_free(void* p, cudaStream_t s) {
    if (p) cudaFreeAsync(p, s);
}

// The contraction (dots == nullptr) or the block-dot test hooks: `fold` selects the
// product's expansion (K-quant codes times their sub-scales) for the hook.
int tcx_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, int32_t* dots,
               cudaStream_t s, bool fold) {
    const char* fn = dots && fold           ? "mmq_debug_product_dots"
                     : fmt == FMT_Q8_0   ? (dots ? "mmq_debug_block_dots_q8_0" : "mmq_gemm_q8_0")
                     : fmt == FMT_Q5_K ? (dots ? "mmq_debug_block_dots_q5_k" : "mmq_gemm_q5_k")
                     : fmt == FMT_Q6_K ? (dots ? "mmq_debug_block_dots_q6_k" : "mmq_gemm_q6_k")
                                       : (dots ? "mmq_debug_block_dots_q4_k" : "mmq_gemm_q4_k");
    if (K % QK_K != 0) {
        report(fn, MMQ_ERR_K_MULTIPLE, "the expanded tensor-core path works in 256-value groups: K % 256 != 0");
        return MMQ_ERR_K_MULTIPLE;
    }
    if ((N + BN - 1) / BN > 65535 || K / QK_K > 65535) {
        report(fn, MMQ_ERR_SHAPE, "N or K too large for the tile grid");
        return MMQ_ERR_SHAPE;
    }
    if (dots && fold)
        return fmt == FMT_Q8_0   ? launch_x<FMT_Q8_0, true, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
               : fmt == FMT_Q5_K ? launch_x<FMT_Q5_K, true, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
               : fmt == FMT_Q6_K ? launch_x<FMT_Q6_K, true, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
                                 : launch_x<FMT_Q4_K, true, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn);
    if (fmt == FMT_Q8_0)
        return dots ? launch_x<FMT_Q8_0, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
                    : launch_x<FMT_Q8_0, false>(nullptr, xq, wq, M, N, K, out, dots, s, fn);
    if (fmt == FMT_Q5_K)
        return dots ? launch_x<FMT_Q5_K, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
                    : launch_x<FMT_Q5_K, false>(nullptr, xq, wq, M, N, K, out, dots, s, fn);
    if (fmt == FMT_Q6_K)
        return dots ? launch_x<FMT_Q6_K, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
                    : launch_x<FMT_Q6_K, false>(nullptr, xq, wq, M, N, K, out, dots, s, fn);
    return dots ? launch_x<FMT_Q4_K, true>(nullptr, xq, wq, M, N, K, out, dots, s, fn)
                : launch_x<FMT_Q4_K, false>(nullptr, xq, wq, M, N, K, out, dots, s, fn);
}

int tcx_linear_launch(int fmt, const float* x, void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                      cudaStream_t s) {
    const char* fn = fmt == FMT_Q8_0   ? "mmq_linear_q8_0"
                     : fmt == FMT_Q5_K ? "mmq_linear_q5_k"
                     : fmt == FMT_Q6_K ? "mmq_linear_q6_k" : "mmq_linear_q4_k";
    if (K % QK_K != 0) {
        report(fn, MMQ_ERR_K_MULTIPLE, "the expanded tensor-core path works in 256-value groups: K % 256 != 0");
        return MMQ_ERR_K_MULTIPLE;
    }
    if ((N + BN - 1) / BN > 65535 || K / QK_K > 65535) {
        report(fn, MMQ_ERR_SHAPE, "N or K too large for the tile grid");
        return MMQ_ERR_SHAPE;
    }
    return fmt == FMT_Q8_0   ? launch_x<FMT_Q8_0, false>(x, xq, wq, M, N, K, out, nullptr, s, fn)
           : fmt == FMT_Q5_K ? launch_x<FMT_Q5_K, false>(x, xq, wq, M, N, K, out, nullptr, s, fn)
           : fmt == FMT_Q6_K ? launch_x<FMT_Q6_K, false>(x, xq, wq, M, N, K, out, nullptr, s, fn)
                             : launch_x<FMT_Q4_K, false>(x, xq, wq, M, N, K, out, nullptr, s, fn);
}

int tcx_launch_noalloc(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                       cudaStream_t s) {
    const char* fn = "mmq_gemm_noalloc";
    if (K % QK_K != 0) {
        report(fn, MMQ_ERR_K_MULTIPLE, "the expanded tensor-core path works in 256-value groups: K % 256 != 0");
        return MMQ_ERR_K_MULTIPLE;
    }
    if ((N + BN - 1) / BN > 65535 || K / QK_K > 65535) {
        report(fn, MMQ_ERR_SHAPE, "N or K too large for the tile grid");
        return MMQ_ERR_SHAPE;
    }
    // the tile width the allocating call picks, unless only 128-wide tiles fit the fixed scratch
    int bn = tcx_tile_n(fmt, M, N);
    if (plan_scratch(fmt, M, N, K, bn, false).total() > NOALLOC_SCRATCH_BYTES) bn = BN;
    if (plan_scratch(fmt, M, N, K, bn, false).total() > NOALLOC_SCRATCH_BYTES) {
        report(fn, MMQ_ERR_SHAPE, "the fixed 64 MiB scratch is too small for this shape");
        return MMQ_ERR_SHAPE;
    }
    // K splits only where their partial outputs fit in the fixed scratch too
    ScratchPlan sp = plan_scratch(fmt, M, N, K, bn);
    if (sp.total() > NOALLOC_SCRATCH_BYTES) sp = plan_scratch(fmt, M, N, K, bn, false);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_CUDA, "cudaGetDevice failed");
        return MMQ_ERR_CUDA;
    }
    uint8_t* ws = noalloc_scratch(dev);
    if (!ws) {
        report(fn, MMQ_ERR_CUDA, "cudaGetSymbolAddress of the fixed scratch failed");
        return MMQ_ERR_CUDA;
    }
    return fmt == FMT_Q8_0   ? launch_bn<FMT_Q8_0, false, true>(bn, nullptr, xq, wq, M, N, K, out, nullptr, ws, sp, s, fn)
           : fmt == FMT_Q5_K ? launch_bn<FMT_Q5_K, false, true>(bn, nullptr, xq, wq, M, N, K, out, nullptr, ws, sp, s, fn)
           : fmt == FMT_Q6_K ? launch_bn<FMT_Q6_K, false, true>(bn, nullptr, xq, wq, M, N, K, out, nullptr, ws, sp, s, fn)
                             : launch_bn<FMT_Q4_K, false, true>(bn, nullptr, xq, wq, M, N, K, out, nullptr, ws, sp, s, fn);
}

// The expert-grouped contraction on the expanded path, after the grouping kernels: one
// expansion launch (the activation tiles gathered through the permutation from xq, and
// the weights of every expert with rows) and the contraction over the tile list, 128-wide
// weight tiles, no K split.
template <int FMT>
int launch_grouped_x(const void* xq, int64_t R, const void* wq, int64_t E, int64_t N, int64_t K, const int2* tiles,
                     const int* ntiles, int64_t max_tiles, const int* offsets, const int* perm, float* out,
                     cudaStream_t s, const char* fn) {
    const int nb = (int)(K / QK), ng = nb / GB;
    const int64_t NTe = (N + BN - 1) / BN;
    static SmemAttr attr;
    const int st_attr = ensure_smem((const void*)k_mmq_tcx<FMT, false, BN, true>, XLayout<FMT, BN>::alloc, attr);
    if (st_attr != MMQ_OK) {
        report(fn, st_attr, "shared-memory request refused");
        return st_attr;
    }
    const size_t b_xa = (size_t)(max_tiles * nb) * XCHUNK, b_ga = (size_t)(max_tiles * ng) * ga_bytes(FMT),
                 b_xb = (size_t)(E * NTe * nb) * wchunk(FMT, BN), b_gw = (size_t)(E * NTe * ng) * gw_bytes(FMT, BN);
    void* ws = nullptr;
    const int st0 = scratch_alloc(b_xa + b_ga + b_xb + b_gw, s, &ws, fn);
    if (st0 != MMQ_OK) return st0;
    uint8_t* xa = static_cast<uint8_t*>(ws);
    uint8_t* ga = xa + b_xa;
    uint8_t* xb = ga + b_ga;
    uint8_t* gw = xb + b_xb;
    const Grouping gp{tiles, ntiles, offsets, perm, (int)NTe};
    const int64_t acts_x = 4 * max_tiles;
    int st = MMQ_OK;
    {
        ProfScope ps("k_expand", s);
        const dim3 eg((unsigned)(acts_x + 4 * E * NTe), (unsigned)ng);
        k_expand<FMT, false, true, false, BN, true><<<eg, EXP_THREADS, 0, s>>>(
            nullptr, static_cast<const uint8_t*>(xq), nullptr, static_cast<const uint8_t*>(wq), (int)R, (int)N, nb,
            (int)acts_x, xa, ga, xb, gw, gp, E * N);
    }
    {
        ProfScope ps("k_mmq_tcx", s);
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)NTe, (unsigned)max_tiles, 1u);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = XLayout<FMT, BN>::alloc;
        cfg.stream = s;
        cudaLaunchAttribute la[1];
        la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        la[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = la;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, k_mmq_tcx<FMT, false, BN, true>, (const uint8_t*)xa,
                                                 (const uint8_t*)ga, (const uint8_t*)xb, (const uint8_t*)gw, (int)R,
                                                 (int)N, nb, out, (int32_t*)nullptr, 0LL, gp);
        if (e != cudaSuccess) {
            cudaGetLastError();
            report(fn, MMQ_ERR_LAUNCH, cudaGetErrorString(e));
            st = MMQ_ERR_LAUNCH;
        }
    }
    if (st == MMQ_OK) st = launch_status(fn);
    scratch_free(ws, s);  // stream-ordered: after the kernels above
    return st;
}

// K splits of the contraction: only when the output has fewer tiles than half the SMs,
// as many as fill the SMs once (at most 8), each at least two 256-value groups.
int tcx_splits(int fmt, int64_t M, int64_t N, int64_t K) {
    const int bn = tcx_tile_n(fmt, M, N);
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
    const int64_t ng = K / QK_K;
    int64_t sp = device_shape().sms / (tiles < 1 ? 1 : tiles);
    if (sp > ng / 2) sp = ng / 2;
    if (sp > 8) sp = 8;
    return sp < 1 ? 1 : (int)sp;
}

// Weight tile width of the contraction.  A CTA's time is about proportional to its
// tile's width, so where the 128-wide tiles leave SMs idle in their last wave (and are
// too many to split K), 96-wide ones are taken when their waves times 96 come to at most
// 0.9 of the 128-wide waves times 128: on 512 x 3584, 152 tiles on the 152 SMs instead of
// 112.
int tcx_tile_n(int fmt, int64_t M, int64_t N) {
    (void)fmt;
    const int64_t sms = device_shape().sms, MT = (M + BM - 1) / BM;
    const int64_t t128 = MT * ((N + BN - 1) / BN), t96 = MT * ((N + 95) / 96);
    if (2 * t128 <= sms) return BN;  // K splits fill the SMs instead
    const int64_t w128 = (t128 + sms - 1) / sms, w96 = (t96 + sms - 1) / sms;
    return 10 * w96 * 96 <= 9 * w128 * BN ? 96 : BN;
}

int tcx_grouped_launch(int fmt, const void* xq, int64_t R, const void* wq, int64_t E, int64_t N, int64_t K,
                       const int2* tiles, const int* ntiles, int64_t max_tiles, const int* offsets, const int* perm,
                       float* out, cudaStream_t s, const char* fn) {
    if (4 * (max_tiles + E * ((N + BN - 1) / BN)) > 0x7fffffff || max_tiles > 65535) {
        report(fn, MMQ_ERR_SHAPE, "too many tiles for the expansion grid");
        return MMQ_ERR_SHAPE;
    }
    return fmt == FMT_Q8_0 ? launch_grouped_x<FMT_Q8_0>(xq, R, wq, E, N, K, tiles, ntiles, max_tiles, offsets, perm, out, s, fn)
           : fmt == FMT_Q5_K
               ? launch_grouped_x<FMT_Q5_K>(xq, R, wq, E, N, K, tiles, ntiles, max_tiles, offsets, perm, out, s, fn)
           : fmt == FMT_Q6_K
               ? launch_grouped_x<FMT_Q6_K>(xq, R, wq, E, N, K, tiles, ntiles, max_tiles, offsets, perm, out, s, fn)
               : launch_grouped_x<FMT_Q4_K>(xq, R, wq, E, N, K, tiles, ntiles, max_tiles, offsets, perm, out, s, fn);
}

int tcx_set_wait_limit(unsigned long long ns) {
    return cudaMemcpyToSymbol(g_tcx_wait_limit_ns, &ns, sizeof(ns)) == cudaSuccess ? MMQ_OK : MMQ_ERR_CUDA;
}

unsigned tcx_take_error() {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tcx_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_tcx_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mmq
