// Tensor-core MMQ for sm_103a: tcgen05.mma into TMEM, with the per-32-block scale
// applied by one fused multiply-add per output element.
//
// The method applies a new f32 scale at every 32-value block boundary ("When the
// Product Won't Collapse", sec. "The obstruction": int8 accumulation is only valid
// inside one constant-scale block), so the int8 block dot D[m,n,b] is formed exactly
// and rescaled in registers ("The viable route is per-backend anyway": apply the scale
// in register, with no shared-memory round trip of the accumulator).
//
// sm_103a has no integer tcgen05 MMA kind, and its int8 mma.sync rate is ~1/12 of the
// fp16 tensor rate.  Every int8 code (and every K-quant code times its 6-bit sub-scale,
// at most 945) is an exact fp16 value, each product is an integer below 2^17 and every
// partial sum of a 32-term block dot an integer below 2^22, so an fp16 x fp16 -> f32
// MMA over one block computes the block dot exactly.
//
// The scale of block b is the outer product S_b = xd[:,b] (x) w[:,b] of two vectors of
// exact f16 values (Q8_0: w = wd; Q4_K, Q5_K: w = d of the super-block, the sub-scale sc_j
// being folded into the weight codes).  A second, K=16 MMA whose operands carry xd and
// w in column 0 (zeros elsewhere) writes S_b exactly into TMEM next to D_b, so the
// epilogue is acc += S_b * D_b: one FMA per element, no scale reads.  The K-quant min term
// sum_j -dmin*m_j*xs_j of a super-block becomes a ninth item with D = sum_j xs_j*m_j
// (K=16 MMA of the f16 sums s against the 6-bit mins) and S = 1 (x) (-dmin)
// ("When Does a Kernel Win Surface?", sec. "Kept levers: Vulkan", affine identity).
//
// Warp roles (one 128 x 128 output tile per CTA, 832 threads):
//   warp 0     TMA producer: raw q8_1 rows (288 B per 256 values) and raw weight rows
//              (Q8_0: 272 B, Q4_K / Q5_K: one 144 / 176 B super-block) for a 256-value k-tile, as
//              2-D tensor copies into a 2-stage ring ("13 . r7-r8 raw-byte MMQ
//              kernel", sec. 2: shared memory holds raw quant bytes; sec. 3.1: whole
//              super-blocks, out-of-range rows zero-filled by the copy engine).
//   warp 1     TMEM owner and MMA issuer: per item, D (two K=16 MMAs; one for a min
//              item) and S (one K=16 MMA) into one of two TMEM slots, then commits.
//   warps 2-9  converters: codes -> exact fp16 (sign-biased byte permute and one half2
//              subtract; Q4_K: half2 fused multiply by sc_j; Q5_K: the fifth bit OR'd in, exact
//              conversion, then a multiply by sc_j) in the canonical K-major
//              no-swizzle UMMA layout, bank-conflict-free; the f16 scale vectors into
//              column 0 of the scale operands.
//   warps 10-25 epilogue, 32 rows x 32 columns each: per item, 16x256b TMEM fragments of
//              D and S, acc += S * D with packed f32x2 FMA; at the end, 8-byte stores.
// Every wait is bounded by wall time; on expiry the kernel records ERR_TIMEOUT, lets
// the other roles fall out, drains its own copies and MMAs, frees TMEM and returns.
// The block-dot test hook (DOTS) stages and multiplies the raw codes (no sc_j fold, no
// min items) through the same pipeline and writes D.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace mmq {
namespace {

using namespace umma;

__device__ unsigned int g_tc_error;

constexpr int BM = 128;                 // activation rows per tile (TMEM lanes)
constexpr int BN = 128;                 // weight rows per tile (MMA N)
constexpr int KT_BLOCKS = 8;            // 32-blocks per staged k-tile (256 values)
constexpr int RS = 2;                   // raw k-tile stages
constexpr int FS = 3;                   // operand slots (one item each)
constexpr int DS = 2;                   // TMEM slots (D and S of one item each)
constexpr int CONV_WARPS = 8;
constexpr int EPI_WARPS = 16;
constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // columns per epilogue warp (4 lane quarters)
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2, WARP_EPI0 = WARP_CONV0 + CONV_WARPS;
constexpr int THREADS = (WARP_EPI0 + EPI_WARPS) * 32;
constexpr int TMEM_COLS = DS * 2 * BN;  // 512: the whole TMEM of the SM
constexpr int A_ROW = KT_BLOCKS * Q8_1_BYTES;  // 288
constexpr int OP_MAIN = BM * QK * 2;    // fp16 tile of one block (K = 32): 8 KiB
constexpr int OP_AUX = BM * 16 * 2;     // fp16 scale operand (K = 16, column 0 used): 4 KiB
constexpr int SLOT = 2 * OP_MAIN + 2 * OP_AUX;

static_assert(BM + BN == 32 * CONV_WARPS, "one scale row (activation or weight) per converter thread");
static_assert(EPI_COLS == 32, "one 16x256b.x4 fragment covers 32 columns");

__host__ __device__ constexpr int b_row(int fmt) { return fmt == FMT_Q8_0 ? KT_BLOCKS * Q8_0_BYTES : kq_bytes(fmt); }
// items per k-tile: 8 blocks, plus the min item of the super-block for Q4_K and Q5_K
__host__ __device__ constexpr int items_per_kt(int fmt, bool dots) {
    return KT_BLOCKS + (is_kquant(fmt) && !dots ? 1 : 0);
}

// barrier indices: raw stages, operand slots (converters -> MMA -> converters), TMEM
// slots (MMA -> epilogue -> MMA), and a drain barrier for teardown
constexpr int BAR_RAW_FULL = 0, BAR_RAW_EMPTY = BAR_RAW_FULL + RS, BAR_SLOT_FULL = BAR_RAW_EMPTY + RS,
              BAR_SLOT_EMPTY = BAR_SLOT_FULL + FS, BAR_D_FULL = BAR_SLOT_EMPTY + FS, BAR_D_EMPTY = BAR_D_FULL + DS,
              BAR_DRAIN = BAR_D_EMPTY + DS, NBARS = BAR_DRAIN + 1;

template <int FMT>
struct Layout {
    static constexpr int rawA = 0;
    static constexpr int rawB = rawA + RS * BM * A_ROW;
    static constexpr int slots = rawB + RS * BN * b_row(FMT);
    static constexpr int sctab = slots + FS * SLOT;  // K-quants: per converter warp, sub-scale pairs of its 64 rows x 8
    static constexpr int bars = sctab + (is_kquant(FMT) ? CONV_WARPS * 32 * 8 * 4 : 0);
    static constexpr int tmem_slot = bars + NBARS * 8;
    static constexpr int total = tmem_slot + 16;
    static constexpr int alloc = total + 1024;  // slack to align the base to 1 KiB
    static_assert(rawB % 1024 == 0 && slots % 1024 == 0 && SLOT % 1024 == 0, "alignment");
    static_assert(alloc <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort) {
    return umma::wait_bar(bar, parity, abort, &g_tc_error);
}
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity) { umma::drain_bar(bar, parity, &g_tc_error); }
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    return umma::warp_wait(bar, parity, abort, &g_tc_error);
}

// GROUPED (expert-grouped contraction): CTA (x, y) takes tile y of a device-built list,
// tiles[y] = (first row in the expert-sorted activations, expert e); its weight rows are
// e * N + n0 .. of the experts' stacked matrices (tmB), rows past row_end[e] belong to
// another expert and are not stored, and row m of the sorted activations is stored to
// output row row_map[m].  CTAs past *ntiles leave at once.
template <int FMT, bool DOTS, bool GROUPED>
__global__ void __launch_bounds__(THREADS, 1)
k_mmq_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N, int nb,
         float* __restrict__ out, int32_t* __restrict__ dots, const int2* __restrict__ tiles,
         const int* __restrict__ ntiles, const int* __restrict__ row_end, const int* __restrict__ row_map) {
    using L = Layout<FMT>;
    constexpr int BROW = b_row(FMT);
    constexpr int IPK = items_per_kt(FMT, DOTS);
    constexpr bool FOLD = is_kquant(FMT) && !DOTS;  // sc_j folded into the weight codes
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    int m0 = blockIdx.y * BM, b0 = n0, mlimit = M;
    if (GROUPED) {
        if ((int)blockIdx.y >= *ntiles) return;  // uniform over the CTA: nothing set up yet
        const int2 tl = tiles[blockIdx.y];
        m0 = tl.x;
        b0 = tl.y * N + n0;
        mlimit = row_end[tl.y];
    }
    const int nkt = nb / KT_BLOCKS;
    const int nitems = nkt * IPK;
    volatile int* abort = &s_abort;
    auto bar = [&](int i) -> uint32_t { return sbase + L::bars + 8 * i; };
    auto slot_ptr = [&](int f) -> uint8_t* { return smem + L::slots + f * SLOT; };

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < RS; ++i) {
            ptx::mbar_init(bar(BAR_RAW_FULL + i), 1);
            ptx::mbar_init(bar(BAR_RAW_EMPTY + i), CONV_WARPS);
        }
        for (int i = 0; i < FS; ++i) {
            ptx::mbar_init(bar(BAR_SLOT_FULL + i), CONV_WARPS);
            ptx::mbar_init(bar(BAR_SLOT_EMPTY + i), 1);
        }
        for (int i = 0; i < DS; ++i) {
            ptx::mbar_init(bar(BAR_D_FULL + i), 1);
            ptx::mbar_init(bar(BAR_D_EMPTY + i), EPI_WARPS);
        }
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        ptx::fence_barrier_init();
    }
    // the scale operands only ever hold column 0: zero all slots once
    for (int i = threadIdx.x; i < FS * 2 * OP_AUX / 16; i += THREADS) {
        const int f = i / (2 * OP_AUX / 16), o = i % (2 * OP_AUX / 16);
        reinterpret_cast<uint4*>(slot_ptr(f) + 2 * OP_MAIN)[o] = make_uint4(0u, 0u, 0u, 0u);
    }
    ptx::fence_proxy_async_smem();
    if (warp == WARP_MMA) {
        ptx::tmem_alloc(sbase + L::tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == WARP_TMA && lane == 0) {
        ptx::tma_prefetch_desc(&tmA);
        ptx::tma_prefetch_desc(&tmB);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::tmem_slot);

    if (warp == WARP_TMA) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint32_t bytes = BM * A_ROW + BN * BROW;
            int issued = 0;
            for (int kt = 0; kt < nkt; ++kt) {
                const int s = kt % RS;
                if (!wait_bar(bar(BAR_RAW_EMPTY + s), ((kt / RS) & 1) ^ 1, abort)) break;
                ptx::mbar_arrive_expect_tx(bar(BAR_RAW_FULL + s), bytes);
                ptx::tma_load_2d(sbase + L::rawA + s * BM * A_ROW, &tmA, bar(BAR_RAW_FULL + s), kt * (A_ROW / 2), m0);
                ptx::tma_load_2d(sbase + L::rawB + s * BN * BROW, &tmB, bar(BAR_RAW_FULL + s), kt * (BROW / 2), b0);
                issued = kt + 1;
            }
            // the copies of the last RS k-tiles may still be in flight after an abort
            for (int kt = issued - RS < 0 ? 0 : issued - RS; kt < issued; ++kt)
                drain_bar(bar(BAR_RAW_FULL + kt % RS), (kt / RS) & 1);
        }
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = make_idesc(BM, BN);
            for (int it = 0; it < nitems; ++it) {
                const int f = it % FS, t = it % DS;
                if (!wait_bar(bar(BAR_SLOT_FULL + f), (it / FS) & 1, abort)) break;
                if (!wait_bar(bar(BAR_D_EMPTY + t), ((it / DS) & 1) ^ 1, abort)) break;
                ptx::tc_fence_after();
                const uint32_t a = sbase + L::slots + f * SLOT, b = a + OP_MAIN;
                const uint32_t as = b + OP_MAIN, bs = as + OP_AUX;
                const uint32_t d = tmem + (uint32_t)(t * 2 * BN), sd = d + BN;
                const bool min_item = IPK > KT_BLOCKS && (it % IPK) == KT_BLOCKS;
                ptx::umma_f16(d, sdesc(a, 512), sdesc(b, 512), idesc, 0u);
                if (!min_item) ptx::umma_f16(d, sdesc(a + 256, 512), sdesc(b + 256, 512), idesc, 1u);
                if (!DOTS) ptx::umma_f16(sd, sdesc(as, 256), sdesc(bs, 256), idesc, 0u);
                ptx::umma_commit(bar(BAR_SLOT_EMPTY + f));
                ptx::umma_commit(bar(BAR_D_FULL + t));
            }
            ptx::umma_commit(bar(BAR_DRAIN));  // arrives once every MMA issued above is done
            drain_bar(bar(BAR_DRAIN), 0);
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ------------------------------------------------------------ converters
        const int cw = warp - WARP_CONV0;
        const int ct = cw * 32 + lane;          // < BM: activation row ct; else weight row ct - BM
        const bool arow = ct < BM;
        const int srow = arow ? ct : ct - BM;
        const int r8 = lane & 7, half = (lane >> 3) & 1, hw = lane >> 4;
        constexpr int UNITS = 32 / CONV_WARPS;   // conversion units per warp and operand
        // Unit i of this warp: 8-row group g = 4i + cw/2, pass p = cw%2.  Its table of the
        // sub-scales of those 32 rows, [8*i + r8][sub-block], is private to the warp.
        uint32_t* sct = reinterpret_cast<uint32_t*>(smem + L::sctab) + cw * 32 * 8;
        bool ok = true;
        int it = 0;
        for (int kt = 0; kt < nkt && ok; ++kt) {
            const int s = kt % RS;
            ok = warp_wait(bar(BAR_RAW_FULL + s), (kt / RS) & 1, abort);
            if (!ok) break;
            const uint8_t* rA = smem + L::rawA + s * BM * A_ROW;
            const uint8_t* rB = smem + L::rawB + s * BN * BROW;
            uint4 whdr = make_uint4(0u, 0u, 0u, 0u);  // K-quants: super-block header of weight row srow
            if (is_kquant(FMT)) {
                if (!arow) whdr = *reinterpret_cast<const uint4*>(rB + srow * BROW);
                if (FOLD) {
                    __syncwarp();  // this warp's reads of the previous k-tile's table are done
                    const int row = 8 * (UNITS * (lane >> 3) + (cw >> 1)) + (lane & 7);  // table row = lane
                    const uint4 h = *reinterpret_cast<const uint4*>(rB + row * BROW);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        int s6, m6;
                        q4_k_scale_min(h.y, h.z, h.w, j, s6, m6);
                        // Q4_K: (sc, -1024 sc) for one fused (1024 + q) * sc - 1024 sc; Q5_K: (sc, sc),
                        // its 5-bit codes converted exactly first ((1024 + q) * sc would overflow)
                        sct[lane * 8 + j] = h2_bits(__halves2half2(
                            __int2half_rn(s6), __int2half_rn(FMT == FMT_Q5_K ? s6 : -1024 * s6)));
                    }
                    __syncwarp();
                }
            }
            for (int ii = 0; ii < IPK && ok; ++ii, ++it) {
                const int f = it % FS;
                const bool block_item = ii < KT_BLOCKS;
                const int j = ii;
                // Raw loads first, then the slot wait, then the stores: the wait's latency
                // overlaps the loads, and no load sits behind a store to the same array.
                // Unit i = (8-row group g, pass p), lane = (hw, half, r8): row 8g + r8
                // takes k-group kg = 2*(p ^ (r8 / 4)) + hw, code word w = 2*kg + half.  Rows
                // r8 and r8 + 4 (same banks: rows are 72 words apart) read different halves
                // of the block, so a load touches 32 different banks; each half-warp stores
                // rows 0-3 of one k-group and rows 4-7 of another, two 64-byte runs in
                // opposite bank halves.
                uint32_t xa[UNITS], wv[UNITS], scv[UNITS];
                uint16_t scol = 0;        // column-0 value of this thread's scale-operand row
                uint32_t mrow[4];         // min item: this thread's A or B row, k = 0..7
                if (block_item) {
#pragma unroll
                    for (int i = 0; i < UNITS; ++i) {
                        const int u = i * CONV_WARPS + cw;
                        const int g = u >> 1, w = 2 * (2 * ((u & 1) ^ (r8 >> 2)) + hw) + half, r = g * 8 + r8;
                        xa[i] = *reinterpret_cast<const uint32_t*>(rA + r * A_ROW + j * Q8_1_BYTES + 4 + w * 4);
                        if (FMT == FMT_Q8_0) {
                            // codes start at an odd half-word for even j: two aligned
                            // words and a funnel shift (for odd j both loads are the same)
                            const int off = r * BROW + j * Q8_0_BYTES + 2 + w * 4;
                            const int sh = (off & 3) * 8;
                            const uint32_t lo = *reinterpret_cast<const uint32_t*>(rB + (off & ~3));
                            const uint32_t hi = *reinterpret_cast<const uint32_t*>(rB + (off & ~3) + (sh ? 4 : 0));
                            wv[i] = __funnelshift_r(lo, hi, sh);
                        } else {
                            const uint32_t raw =
                                *reinterpret_cast<const uint32_t*>(rB + r * BROW + kq_qs_off(FMT) + 32 * (j >> 1) + w * 4);
                            wv[i] = (j & 1) ? ((raw >> 4) & 0x0F0F0F0Fu) : (raw & 0x0F0F0F0Fu);
                            if (FMT == FMT_Q5_K) {  // fifth bit of values 4w .. 4w + 3: bit j of high-bit bytes
                                const uint32_t qh = *reinterpret_cast<const uint32_t*>(rB + r * BROW + 16 + w * 4);
                                wv[i] |= ((qh >> j) & 0x01010101u) << 4;
                            }
                            if (FOLD) scv[i] = sct[(i * 8 + r8) * 8 + j];  // table row 8i + r8 is row 8g + r8
                        }
                    }
                    if (arow)
                        scol = *reinterpret_cast<const uint16_t*>(rA + srow * A_ROW + j * Q8_1_BYTES);  // xd
                    else if (FMT == FMT_Q8_0)
                        scol = *reinterpret_cast<const uint16_t*>(rB + srow * BROW + j * Q8_0_BYTES);   // wd
                    else
                        scol = (uint16_t)(whdr.x & 0xffffu);                                            // d
                } else {
                    // K-quant min item: A row m = (s of the 8 blocks, 0 x 8), B row n = (m_0..m_7,
                    // 0 x 8); scale operands: A = 1, B = -dmin
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        if (arow) {
                            const uint32_t s0 = *reinterpret_cast<const uint32_t*>(rA + srow * A_ROW + (2 * jj) * Q8_1_BYTES);
                            const uint32_t s1 =
                                *reinterpret_cast<const uint32_t*>(rA + srow * A_ROW + (2 * jj + 1) * Q8_1_BYTES);
                            mrow[jj] = (s0 >> 16) | (s1 & 0xffff0000u);
                        } else {
                            int sc0, mn0, sc1, mn1;
                            q4_k_scale_min(whdr.y, whdr.z, whdr.w, 2 * jj, sc0, mn0);
                            q4_k_scale_min(whdr.y, whdr.z, whdr.w, 2 * jj + 1, sc1, mn1);
                            mrow[jj] = h2_bits(__halves2half2(__int2half_rn(mn0), __int2half_rn(mn1)));
                        }
                    }
                    scol = arow ? (uint16_t)0x3C00u : (uint16_t)((whdr.x >> 16) ^ 0x8000u);  // 1.0 / -dmin
                }
                ok = warp_wait(bar(BAR_SLOT_EMPTY + f), ((it / FS) & 1) ^ 1, abort);
                if (!ok) break;
                uint8_t* oA = slot_ptr(f);
                uint8_t* oB = oA + OP_MAIN;
                uint16_t* aux = reinterpret_cast<uint16_t*>(oB + OP_MAIN + (arow ? 0 : OP_AUX));
                if (block_item) {
#pragma unroll
                    for (int i = 0; i < UNITS; ++i) {
                        const int u = i * CONV_WARPS + cw;
                        const int g = u >> 1, w = 2 * (2 * ((u & 1) ^ (r8 >> 2)) + hw) + half;
                        const int dst = g * 512 + (w >> 1) * 128 + r8 * 16 + half * 8;
                        *reinterpret_cast<uint2*>(oA + dst) = i8x4_to_f16x4(xa[i]);
                        if (FMT == FMT_Q8_0)
                            *reinterpret_cast<uint2*>(oB + dst) = i8x4_to_f16x4(wv[i]);
                        else if (FOLD && FMT == FMT_Q5_K) {
                            const uint2 c = u4x4_scaled_f16x4(wv[i], __float2half2_rn(1.f), __float2half2_rn(-1024.f));
                            const __half2 sc2 = __low2half2(bits_h2(scv[i]));
                            *reinterpret_cast<uint2*>(oB + dst) =
                                make_uint2(h2_bits(__hmul2(bits_h2(c.x), sc2)), h2_bits(__hmul2(bits_h2(c.y), sc2)));
                        } else if (FOLD)
                            *reinterpret_cast<uint2*>(oB + dst) = u4x4_scaled_f16x4(
                                wv[i], __low2half2(bits_h2(scv[i])), __high2half2(bits_h2(scv[i])));
                        else
                            *reinterpret_cast<uint2*>(oB + dst) =
                                u4x4_scaled_f16x4(wv[i], __float2half2_rn(1.f), __float2half2_rn(-1024.f));
                    }
                } else {
                    uint8_t* o = arow ? oA : oB;
                    *reinterpret_cast<uint4*>(o + core_off(srow, 0, 512)) = make_uint4(mrow[0], mrow[1], mrow[2], mrow[3]);
                    *reinterpret_cast<uint4*>(o + core_off(srow, 1, 512)) = make_uint4(0u, 0u, 0u, 0u);
                }
                aux[core_off(srow, 0, 256) / 2] = scol;
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BAR_SLOT_FULL + f));
            }
            __syncwarp();
            if (ok && lane == 0) ptx::mbar_arrive(bar(BAR_RAW_EMPTY + s));
        }
    } else {
        // ------------------------------------------------------------ epilogue
        epilogue_128x128<DOTS, DS, BN, false>(warp & 3, (warp - WARP_EPI0) >> 2, lane, tmem, nitems, bar(BAR_D_FULL),
                                              bar(BAR_D_EMPTY), abort, &g_tc_error, mlimit, N, m0, n0, nb, out, dots,
                                              GROUPED ? row_map : nullptr);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

bool make_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
              uint32_t box_rows) {
    return make_byte_map(map, base, row_bytes, rows, box_bytes, box_rows, 2);
}

template <int FMT, bool DOTS>
int launch_t(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, int32_t* dots,
             cudaStream_t s, const char* fn) {
    const int nb = (int)(K / QK);
    CUtensorMap ta, tb;
    if (!make_map(&ta, xq, (uint64_t)nb * Q8_1_BYTES, (uint64_t)M, A_ROW, BM) ||
        !make_map(&tb, wq, (uint64_t)(FMT == FMT_Q8_0 ? nb * Q8_0_BYTES : nb / 8 * kq_bytes(FMT)), (uint64_t)N,
                  b_row(FMT), BN)) {
        report(fn, MMQ_ERR_CUDA, "tensor map encoding failed");
        return MMQ_ERR_CUDA;
    }
    const int smem = Layout<FMT>::alloc;
    static SmemAttr attr;
    const int e_attr = ensure_smem((const void*)k_mmq_tc<FMT, DOTS, false>, smem, attr);
    if (e_attr != MMQ_OK) {
        report(fn, e_attr, "shared-memory request refused");
        return e_attr;
    }
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    {
        ProfScope ps("k_mmq_tc", s);
        k_mmq_tc<FMT, DOTS, false><<<grid, THREADS, smem, s>>>(ta, tb, (int)M, (int)N, nb, out, dots, nullptr, nullptr,
                                                               nullptr, nullptr);
    }
    return launch_status(fn);
}

// The grouped contraction over the expert-sorted activations xs (R rows): grid (N tiles,
// max_tiles), tiles / ntiles / row_end / row_map built on the device by the grouping
// kernels (grouped.cu).
template <int FMT>
int launch_grouped_t(const void* xs, const void* wq, int64_t R, int64_t E, int64_t N, int64_t K, const int2* tiles,
                     const int* ntiles, int64_t max_tiles, const int* row_end, const int* row_map, float* out,
                     cudaStream_t s, const char* fn) {
    const int nb = (int)(K / QK);
    CUtensorMap ta, tb;
    if (!make_map(&ta, xs, (uint64_t)nb * Q8_1_BYTES, (uint64_t)R, A_ROW, BM) ||
        !make_map(&tb, wq, (uint64_t)(FMT == FMT_Q8_0 ? nb * Q8_0_BYTES : nb / 8 * kq_bytes(FMT)), (uint64_t)(E * N),
                  b_row(FMT), BN)) {
        report(fn, MMQ_ERR_CUDA, "tensor map encoding failed");
        return MMQ_ERR_CUDA;
    }
    const int smem = Layout<FMT>::alloc;
    static SmemAttr attr;
    const int e_attr = ensure_smem((const void*)k_mmq_tc<FMT, false, true>, smem, attr);
    if (e_attr != MMQ_OK) {
        report(fn, e_attr, "shared-memory request refused");
        return e_attr;
    }
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)max_tiles);
    {
        ProfScope ps("k_mmq_tc_grouped", s);
        k_mmq_tc<FMT, false, true><<<grid, THREADS, smem, s>>>(ta, tb, (int)R, (int)N, nb, out, nullptr, tiles, ntiles,
                                                               row_end, row_map);
    }
    return launch_status(fn);
}

}  // namespace

int tc_grouped_launch(int fmt, const void* xs, const void* wq, int64_t R, int64_t E, int64_t N, int64_t K,
                      const int2* tiles, const int* ntiles, int64_t max_tiles, const int* row_end, const int* row_map,
                      float* out, cudaStream_t s) {
    const char* fn = fmt == FMT_Q8_0   ? "mmq_gemm_grouped_q8_0"
                     : fmt == FMT_Q5_K ? "mmq_gemm_grouped_q5_k" : "mmq_gemm_grouped_q4_k";
    if (fmt == FMT_Q8_0)
        return launch_grouped_t<FMT_Q8_0>(xs, wq, R, E, N, K, tiles, ntiles, max_tiles, row_end, row_map, out, s, fn);
    if (fmt == FMT_Q5_K)
        return launch_grouped_t<FMT_Q5_K>(xs, wq, R, E, N, K, tiles, ntiles, max_tiles, row_end, row_map, out, s, fn);
    return launch_grouped_t<FMT_Q4_K>(xs, wq, R, E, N, K, tiles, ntiles, max_tiles, row_end, row_map, out, s, fn);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A byte matrix of `rows` rows of `row_bytes` (a multiple of 16) viewed as elements of
// `elem_bytes` (2 or 8) for the copy engine; box = box_bytes x box_rows, out-of-range
// reads zero-filled.
bool make_byte_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                   uint32_t box_rows, int elem_bytes) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {row_bytes / (uint64_t)elem_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_bytes / (uint32_t)elem_bytes, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, elem_bytes == 8 ? CU_TENSOR_MAP_DATA_TYPE_UINT64 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_available() { return true; }

int tc_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, int32_t* dots,
              cudaStream_t s) {
    const char* fn = fmt == FMT_Q8_0   ? (dots ? "mmq_debug_block_dots_q8_0" : "mmq_gemm_q8_0")
                     : fmt == FMT_Q5_K ? (dots ? "mmq_debug_block_dots_q5_k" : "mmq_gemm_q5_k")
                     : fmt == FMT_Q6_K ? (dots ? "mmq_debug_block_dots_q6_k" : "mmq_gemm_q6_k")
                                       : (dots ? "mmq_debug_block_dots_q4_k" : "mmq_gemm_q4_k");
    if (fmt == FMT_Q6_K) {  // its 210-byte rows are not 16-byte strided: no 2-D tensor copies
        report(fn, MMQ_ERR_ARG, "the converter tensor-core kernel takes Q8_0, Q4_K and Q5_K (Q6_K: the expanded path)");
        return MMQ_ERR_ARG;
    }
    if (K % QK_K != 0) {
        report(fn, MMQ_ERR_K_MULTIPLE, "the tensor-core path stages 256-value k-tiles: K % 256 != 0");
        return MMQ_ERR_K_MULTIPLE;
    }
    if ((M + BM - 1) / BM > 65535) {
        report(fn, MMQ_ERR_SHAPE, "M too large for the tile grid");
        return MMQ_ERR_SHAPE;
    }
    if (fmt == FMT_Q8_0)
        return dots ? launch_t<FMT_Q8_0, true>(xq, wq, M, N, K, out, dots, s, fn)
                    : launch_t<FMT_Q8_0, false>(xq, wq, M, N, K, out, dots, s, fn);
    if (fmt == FMT_Q5_K)
        return dots ? launch_t<FMT_Q5_K, true>(xq, wq, M, N, K, out, dots, s, fn)
                    : launch_t<FMT_Q5_K, false>(xq, wq, M, N, K, out, dots, s, fn);
    return dots ? launch_t<FMT_Q4_K, true>(xq, wq, M, N, K, out, dots, s, fn)
                : launch_t<FMT_Q4_K, false>(xq, wq, M, N, K, out, dots, s, fn);
}

unsigned tc_take_error() {
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(v)) != cudaSuccess) return 0;
    if (v) {
        const unsigned zero = 0;
        cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(zero));
    }
    return v;
}

}  // namespace mmq
