// Tensor-core MMQ for sm_103a: tcgen05.mma into TMEM with a per-32-block drain.
//
// The method applies a new f32 scale at every 32-value block boundary ("When the
// Product Won't Collapse", sec. "The obstruction": int8 accumulation is only valid
// inside one constant-scale block), so the int8 block dot D[m,n,b] must be formed
// exactly, then rescaled in registers ("The viable route is per-backend anyway": apply
// the scale in register, with no shared-memory round trip of the accumulator).
//
// sm_103a has no integer tcgen05 MMA kind, and its int8 mma.sync rate is ~1/12 of the
// fp16 tensor rate.  Every int8 code (and every Q4_K nibble) is an exact fp16 value,
// each product is an integer of magnitude <= 2^14 and every partial sum of a 32-term
// block dot is an integer of magnitude <= 2^19, so an fp16 x fp16 -> f32 MMA over one
// block computes D exactly.  That is the contraction used here.
//
// Warp roles (one 128 x 128 output tile per CTA, 704 threads):
//   warp 0     TMA producer: raw q8_1 rows (288 B per 256 values) and raw weight rows
//              (Q8_0: 272 B, Q4_K: one 144 B super-block) for a 256-value k-tile, as
//              2-D tensor copies into a 2-stage ring ("13 . r7-r8 raw-byte MMQ
//              kernel", sec. 2: shared memory holds raw quant bytes; sec. 3.1: whole
//              super-blocks, out-of-range rows zero-filled by the copy engine).
//   warp 1     TMEM owner and MMA issuer: per 32-block, two K=16 MMAs (M=128, N=128)
//              into one of four TMEM accumulators; one tcgen05.commit per group of
//              two blocks (barrier round trips cost more than the work between them).
//   warps 2-5  converters: codes -> fp16 (sign-biased byte permute + one half2
//              subtract, exact) into the canonical K-major no-swizzle UMMA layout, and
//              the per-row / per-column block scales into a small scale ring
//              (Q4_K: d*sc_j and dmin*m_j from the 12 packed bytes, computed once per
//              (row, block) instead of per lane, as in sec. 3.2 of the same page).
//   warps 6-21 epilogue, 32 rows x 32 columns each: per 32-block, tcgen05.ld of the
//              f32 block dots in 8-column chunks (the next loads while one is rescaled), then
//              acc += (xd*wd) * D (Q4_K: wd = d*sc_j, and acc -= dmin*m_j*xs) with packed
//              f32x2 multiply / FMA in registers; at the end the tile is stored to out.
// Every wait is bounded by wall time; on expiry the kernel records ERR_TIMEOUT, lets
// the other roles fall out, drains its own copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mmq {
namespace {

__device__ unsigned int g_tc_error;

constexpr int BM = 128;                 // activation rows per tile (TMEM lanes)
constexpr int BN = 128;                 // weight rows per tile (MMA N, TMEM columns)
constexpr int KT_BLOCKS = 8;            // 32-blocks per staged k-tile (256 values)
constexpr int RS = 2;                   // raw k-tile stages
constexpr int FS = 4;                   // fp16 operand slots (one 32-block each)
constexpr int SCN = 8;                  // scale slots (one 32-block each)
constexpr int DS = 4;                   // TMEM accumulators (one 32-block each)
constexpr int G = 2;                    // 32-blocks per barrier round trip (a "group")
constexpr int SG = FS / G;              // operand slot groups in flight
constexpr int SCG = SCN / G;            // scale slot groups in flight
constexpr int DG = DS / G;              // TMEM groups in flight
constexpr int CONV_WARPS = 4;
constexpr int EPI_WARPS = 16;
constexpr int EPI_COLS = BN / (EPI_WARPS / 4);  // columns per epilogue warp (4 lane quarters)
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2, WARP_EPI0 = WARP_CONV0 + CONV_WARPS;
constexpr int THREADS = (WARP_EPI0 + EPI_WARPS) * 32;
constexpr int TMEM_COLS = DS * BN;      // 512: the whole TMEM of the SM
constexpr int A_ROW = KT_BLOCKS * Q8_1_BYTES;  // 288
constexpr int OP_A = BM * QK * 2;       // fp16 A tile of one block: 8 KiB
constexpr int OP_B = BN * QK * 2;       // fp16 B tile of one block: 8 KiB
constexpr int SC_FLOATS = 2 * BM + 2 * BN;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // bound on any one wait
constexpr uint32_t WAIT_SLEEP_NS = 100000;           // longest sleep inside one poll

static_assert(BM == 32 * CONV_WARPS && BN == 32 * CONV_WARPS, "one activation and one weight scale row per converter thread");
static_assert(32 % CONV_WARPS == 0, "32 conversion units per operand tile");
static_assert(EPI_WARPS % 4 == 0 && EPI_COLS % 8 == 0, "epilogue covers 4 lane quarters x column groups");

__host__ __device__ constexpr int b_row(int fmt) { return fmt == FMT_Q8_0 ? KT_BLOCKS * Q8_0_BYTES : Q4_K_BYTES; }

// barrier indices.  A slot group holds the fp16 operands of G 32-blocks (SLOT_FULL:
// every converter warp arrives; SLOT_EMPTY: the MMA commit).  The scales of a group sit
// in a deeper ring of their own (SC_FULL: converters; SC_EMPTY: every epilogue warp), so
// that operand slots come free as soon as their MMAs complete.  D_FULL / D_EMPTY guard
// the G TMEM accumulators of a group.
constexpr int BAR_RAW_FULL = 0, BAR_RAW_EMPTY = BAR_RAW_FULL + RS, BAR_SLOT_FULL = BAR_RAW_EMPTY + RS,
              BAR_SLOT_EMPTY = BAR_SLOT_FULL + SG, BAR_SC_FULL = BAR_SLOT_EMPTY + SG, BAR_SC_EMPTY = BAR_SC_FULL + SCG,
              BAR_D_FULL = BAR_SC_EMPTY + SCG, BAR_D_EMPTY = BAR_D_FULL + DG, BAR_DRAIN = BAR_D_EMPTY + DG,
              NBARS = BAR_DRAIN + 1;
static_assert(KT_BLOCKS % G == 0 && FS % G == 0 && DS % G == 0 && SCN % G == 0, "groups tile the rings");

template <int FMT>
struct Layout {
    static constexpr int rawA = 0;
    static constexpr int rawB = rawA + RS * BM * A_ROW;
    static constexpr int opA = rawB + RS * BN * b_row(FMT);
    static constexpr int opB = opA + FS * OP_A;
    static constexpr int sc = opB + FS * OP_B;
    static constexpr int bars = sc + SCN * SC_FLOATS * 4;
    static constexpr int tmem_slot = bars + NBARS * 8;
    static constexpr int total = tmem_slot + 16;
    static constexpr int alloc = total + 1024;  // slack to align the base to 1 KiB
    static_assert(rawB % 1024 == 0 && opA % 1024 == 0 && opB % 1024 == 0 && sc % 16 == 0, "alignment");
};

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of 8 rows x 16 B
// (8 fp16 along K) stored as 128 contiguous bytes; the next core matrix along K is
// 128 B further (leading-dimension offset), the next 8-row group 512 B further
// (stride-dimension offset: 4 core matrices cover the block's 32 values of K).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(512 >> 4) << 32) |
           (1ull << 46);
}

__device__ __forceinline__ uint32_t h2_sub_bits(uint32_t a, uint32_t b) {
    __half2 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __half2 r = __hsub2(x, y);
    uint32_t o;
    memcpy(&o, &r, 4);
    return o;
}

// Four signed int8 codes -> four exact fp16 values.  (x + 128) is placed in the low
// mantissa byte of 1024.0 (bits 0x64xx), then 1152 = 1024 + 128 is subtracted.
__device__ __forceinline__ uint2 i8x4_to_f16x4(uint32_t w) {
    const uint32_t u = w ^ 0x80808080u;
    return make_uint2(h2_sub_bits(__byte_perm(u, 0x64646464u, 0x4140), 0x64806480u),
                      h2_sub_bits(__byte_perm(u, 0x64646464u, 0x4342), 0x64806480u));
}

// Four codes 0..15 (one per byte) -> four exact fp16 values (1024 + q, minus 1024).
__device__ __forceinline__ uint2 u4x4_to_f16x4(uint32_t w) {
    return make_uint2(h2_sub_bits(__byte_perm(w, 0x64646464u, 0x4140), 0x64006400u),
                      h2_sub_bits(__byte_perm(w, 0x64646464u, 0x4342), 0x64006400u));
}

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting or the wall
// time limit ran out (then the error word and the abort flag are set).  Inlined: a
// call here costs the waiting warp more than the wait itself.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
        if (ptx::mbar_try_wait_sleep(bar, parity, WAIT_SLEEP_NS)) return true;
        if (*abort) return false;
        if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(&g_tc_error, ERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// Teardown wait: bounded by time only (used to drain in-flight copies and MMAs).
__device__ __noinline__ void drain_bar(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
            atomicOr(&g_tc_error, ERR_TIMEOUT);
            return;
        }
    }
}

// Lane 0 polls (one shared-memory barrier access per poll instead of 32); the other
// lanes take its answer, so the warp stays on one path.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    int ok = 0;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort);
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

template <int FMT, bool DOTS>
__global__ void __launch_bounds__(THREADS, 1)
k_mmq_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, int M, int N, int nb,
         float* __restrict__ out, int32_t* __restrict__ dots) {
    using L = Layout<FMT>;
    constexpr int BROW = b_row(FMT);
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_abort;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = ptx::smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
    const int nkt = nb / KT_BLOCKS;
    volatile int* abort = &s_abort;
    auto bar = [&](int i) -> uint32_t { return sbase + L::bars + 8 * i; };

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < RS; ++i) {
            ptx::mbar_init(bar(BAR_RAW_FULL + i), 1);
            ptx::mbar_init(bar(BAR_RAW_EMPTY + i), CONV_WARPS);
        }
        for (int i = 0; i < SG; ++i) {
            ptx::mbar_init(bar(BAR_SLOT_FULL + i), CONV_WARPS);
            ptx::mbar_init(bar(BAR_SLOT_EMPTY + i), 1);
        }
        for (int i = 0; i < SCG; ++i) {
            ptx::mbar_init(bar(BAR_SC_FULL + i), CONV_WARPS);
            ptx::mbar_init(bar(BAR_SC_EMPTY + i), EPI_WARPS);
        }
        for (int i = 0; i < DG; ++i) {
            ptx::mbar_init(bar(BAR_D_FULL + i), 1);
            ptx::mbar_init(bar(BAR_D_EMPTY + i), EPI_WARPS);
        }
        ptx::mbar_init(bar(BAR_DRAIN), 1);
        ptx::fence_barrier_init();
    }
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
    const int ng = nb / G;

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
                ptx::tma_load_2d(sbase + L::rawB + s * BN * BROW, &tmB, bar(BAR_RAW_FULL + s), kt * (BROW / 2), n0);
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
            for (int gi = 0; gi < ng; ++gi) {
                const int gs = gi % SG, gd = gi % DG;
                if (!wait_bar(bar(BAR_SLOT_FULL + gs), (gi / SG) & 1, abort)) break;
                if (!wait_bar(bar(BAR_D_EMPTY + gd), ((gi / DG) & 1) ^ 1, abort)) break;
                ptx::tc_fence_after();
#pragma unroll
                for (int jj = 0; jj < G; ++jj) {
                    const int bi = gi * G + jj, f = bi % FS, t = bi % DS;
                    const uint32_t a = sbase + L::opA + f * OP_A, b = sbase + L::opB + f * OP_B;
                    const uint32_t d = tmem + (uint32_t)(t * BN);
                    ptx::umma_f16(d, sdesc(a), sdesc(b), idesc, 0u);
                    ptx::umma_f16(d, sdesc(a + 256), sdesc(b + 256), idesc, 1u);
                }
                ptx::umma_commit(bar(BAR_SLOT_EMPTY + gs));
                ptx::umma_commit(bar(BAR_D_FULL + gd));
            }
            ptx::umma_commit(bar(BAR_DRAIN));  // arrives once every MMA issued above is done
            drain_bar(bar(BAR_DRAIN), 0);
        }
        __syncwarp();
    } else if (warp < WARP_EPI0) {
        // ------------------------------------------------------------ converters
        const int cw = warp - WARP_CONV0;
        const int ct = cw * 32 + lane;
        const int r8 = lane & 7, half = (lane >> 3) & 1, hw = lane >> 4;
        bool ok = true;
        for (int kt = 0; kt < nkt && ok; ++kt) {
            const int s = kt % RS;
            ok = warp_wait(bar(BAR_RAW_FULL + s), (kt / RS) & 1, abort);
            if (!ok) break;
            const uint8_t* rA = smem + L::rawA + s * BM * A_ROW;
            const uint8_t* rB = smem + L::rawB + s * BN * BROW;
            for (int gl = 0; gl < KT_BLOCKS / G; ++gl) {
                const int gi = kt * (KT_BLOCKS / G) + gl, gs = gi % SG, gc = gi % SCG;
                ok = warp_wait(bar(BAR_SLOT_EMPTY + gs), ((gi / SG) & 1) ^ 1, abort) &&
                     warp_wait(bar(BAR_SC_EMPTY + gc), ((gi / SCG) & 1) ^ 1, abort);
                if (!ok) break;
#pragma unroll 1
                for (int jj = 0; jj < G; ++jj) {
                    const int j = gl * G + jj, bi = kt * KT_BLOCKS + j, f = bi % FS;
                    uint8_t* oA = smem + L::opA + f * OP_A;
                    uint8_t* oB = smem + L::opB + f * OP_B;
                    float* sc = reinterpret_cast<float*>(smem + L::sc + (bi % SCN) * SC_FLOATS * 4);
                    // All raw loads first (the stores below go to the same shared array,
                    // so the compiler would otherwise keep every load behind the previous
                    // store).  Unit i = (8-row group g, pass p), lane = (hw, half, r8):
                    // row 8g + r8 takes k-group kg = 2*(p ^ (r8 / 4)) + hw, code word
                    // w = 2*kg + half.  Rows r8 and r8 + 4 (same banks: rows are 72 words
                    // apart) read different halves of the block, so a load touches 32
                    // different banks; each half-warp stores rows 0-3 of one k-group and
                    // rows 4-7 of another, two 64-byte runs in opposite bank halves.
                    constexpr int UNITS = 32 / CONV_WARPS;
                    uint32_t xa[UNITS], wv[UNITS];
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
                                *reinterpret_cast<const uint32_t*>(rB + r * BROW + 16 + 32 * (j >> 1) + w * 4);
                            wv[i] = (j & 1) ? ((raw >> 4) & 0x0F0F0F0Fu) : (raw & 0x0F0F0F0Fu);
                        }
                    }
                    // scales: converter thread ct takes activation row ct and weight row ct
                    const uint32_t hd = *reinterpret_cast<const uint32_t*>(rA + ct * A_ROW + j * Q8_1_BYTES);
                    float wsc, wmn;
                    if (FMT == FMT_Q8_0) {
                        wsc = f16_bits_to_f32(
                            *reinterpret_cast<const unsigned short*>(rB + ct * BROW + j * Q8_0_BYTES));
                        wmn = 0.f;
                    } else {
                        const uint4 p = *reinterpret_cast<const uint4*>(rB + ct * BROW);
                        int s6, m6;
                        q4_k_scale_min(p.y, p.z, p.w, j, s6, m6);
                        wsc = f16_bits_to_f32(p.x) * (float)s6;        // exact: d * sc_j
                        wmn = f16_bits_to_f32(p.x >> 16) * (float)m6;  // exact: dmin * m_j
                    }
#pragma unroll
                    for (int i = 0; i < UNITS; ++i) {
                        const int u = i * CONV_WARPS + cw;
                        const int g = u >> 1, w = 2 * (2 * ((u & 1) ^ (r8 >> 2)) + hw) + half;
                        const int dst = g * 512 + (w >> 1) * 128 + r8 * 16 + half * 8;
                        *reinterpret_cast<uint2*>(oA + dst) = i8x4_to_f16x4(xa[i]);
                        *reinterpret_cast<uint2*>(oB + dst) =
                            FMT == FMT_Q8_0 ? i8x4_to_f16x4(wv[i]) : u4x4_to_f16x4(wv[i]);
                    }
                    // layout: xd[BM], -xs[BM], w[BN], wmin[BN]
                    sc[ct] = f16_bits_to_f32(hd);
                    sc[BM + ct] = -f16_bits_to_f32(hd >> 16);  // -xs, for the min term
                    sc[2 * BM + ct] = wsc;
                    sc[2 * BM + BN + ct] = wmn;
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(bar(BAR_SLOT_FULL + gs));
                    ptx::mbar_arrive(bar(BAR_SC_FULL + gc));
                }
            }
            __syncwarp();
            if (ok && lane == 0) ptx::mbar_arrive(bar(BAR_RAW_EMPTY + s));
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Warp (q = lane quarter, cg = column group) owns rows 32q..32q+31 and columns
        // c0..c0+31 of the tile.  The block dots are read as two 16-lane x 32-column
        // fragments: thread t holds rows 32q + t/4 + {0, 8, 16, 24} and columns
        // c0 + 8k + 2*(t%4) + {0, 1}, k = 0..3, so it needs 4 row scales and 8 column
        // scales per block (a one-row-per-thread layout would need all 32 column scales,
        // each a broadcast read of shared memory).
        const int q = warp & 3;
        const int cg = (warp - WARP_EPI0) >> 2;
        const int c0 = cg * EPI_COLS;
        const int tr = lane >> 2, tc2 = 2 * (lane & 3);
        const int rloc0 = 32 * q + tr;                 // rows rloc0 + 8*i, i = 0..3 (i = 2*half + i2)
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0;
        static_assert(EPI_COLS == 32, "one 16x256b.x4 fragment covers 32 columns");
        unsigned long long acc[16];                    // [row i][col pair k] as packed pairs
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] = 0ull;
        for (int gi = 0; gi < ng; ++gi) {
            const int gc = gi % SCG, gd = gi % DG;
            if (!(warp_wait(bar(BAR_D_FULL + gd), (gi / DG) & 1, abort) &&
                  warp_wait(bar(BAR_SC_FULL + gc), (gi / SCG) & 1, abort)))
                break;
            ptx::tc_fence_after();
#pragma unroll 1
            for (int jj = 0; jj < G; ++jj) {
                const int bi = gi * G + jj, t = bi % DS;
                const float* sc = reinterpret_cast<const float*>(smem + L::sc + (bi % SCN) * SC_FLOATS * 4);
                const uint32_t taddr = lane_base + (uint32_t)(t * BN);
                if (DOTS) {
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t dv[16];
                        ptx::tmem_ld16x256b_x4(taddr + ((uint32_t)(16 * hh) << 16), dv);
                        ptx::tmem_ld_wait(dv);
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int mrow = m0 + rloc0 + 16 * hh + 8 * i;
#pragma unroll
                            for (int k = 0; k < 4; ++k)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const int n = n0 + c0 + 8 * k + tc2 + e;
                                    if (mrow < M && n < N)
                                        dots[((long long)mrow * N + n) * nb + bi] =
                                            __float2int_rn(__uint_as_float(dv[4 * k + 2 * i + e]));
                                }
                        }
                    }
                } else {
                    // column scales (and, for Q4_K, column min scales) of this thread
                    unsigned long long w2[4], wm2[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        w2[k] = *reinterpret_cast<const unsigned long long*>(sc + 2 * BM + c0 + 8 * k + tc2);
                        if (FMT == FMT_Q4_K)
                            wm2[k] = *reinterpret_cast<const unsigned long long*>(sc + 2 * BM + BN + c0 + 8 * k + tc2);
                    }
                    // acc[row i][pair k] += (xd_i * w_k) * D  (Q4_K: += -xs_i * wmin_k)
                    auto rescale = [&](const uint32_t (&dv)[16], int hh) {
#pragma unroll
                        for (int i2 = 0; i2 < 2; ++i2) {
                            const int i = 2 * hh + i2;
                            const float xd = sc[rloc0 + 8 * i];
                            const unsigned long long xd2 = ptx::f2_bits(xd, xd);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const unsigned long long dd = ptx::f2_bits(__uint_as_float(dv[4 * k + 2 * i2]),
                                                                           __uint_as_float(dv[4 * k + 2 * i2 + 1]));
                                acc[4 * i + k] = ptx::fma_f32x2(ptx::mul_f32x2(xd2, w2[k]), dd, acc[4 * i + k]);
                            }
                            if (FMT == FMT_Q4_K) {
                                const float nxs = sc[BM + rloc0 + 8 * i];
                                const unsigned long long nxs2 = ptx::f2_bits(nxs, nxs);
#pragma unroll
                                for (int k = 0; k < 4; ++k) acc[4 * i + k] = ptx::fma_f32x2(nxs2, wm2[k], acc[4 * i + k]);
                            }
                        }
                    };
                    // the two 16-lane halves one after the other (keeping both in flight
                    // costs 16 more registers than the budget of 704 threads allows)
                    uint32_t d0[16];
                    ptx::tmem_ld16x256b_x4(taddr, d0);
                    ptx::tmem_ld_wait(d0);
                    rescale(d0, 0);
                    ptx::tmem_ld16x256b_x4(taddr + (16u << 16), d0);
                    ptx::tmem_ld_wait(d0);
                    rescale(d0, 1);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(bar(BAR_D_EMPTY + gd));
                ptx::mbar_arrive(bar(BAR_SC_EMPTY + gc));
            }
        }
        if (!DOTS && !*abort) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int mrow = m0 + rloc0 + 8 * i;
                if (mrow >= M) continue;
                float* orow = out + (long long)mrow * N;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int n = n0 + c0 + 8 * k + tc2;
                    if (n + 1 < N && (N & 1) == 0) {
                        *reinterpret_cast<unsigned long long*>(orow + n) = acc[4 * i + k];
                    } else {
                        if (n < N) orow[n] = __uint_as_float((uint32_t)acc[4 * i + k]);
                        if (n + 1 < N) orow[n + 1] = __uint_as_float((uint32_t)(acc[4 * i + k] >> 32));
                    }
                }
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == WARP_MMA) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
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

// A byte matrix of `rows` rows of `row_bytes` (even, multiple of 16) viewed as u16 for
// the copy engine, box = box_bytes x box_rows.
bool make_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
              uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {row_bytes / 2, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_bytes / 2, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int FMT, bool DOTS>
int launch_t(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, int32_t* dots,
             cudaStream_t s, const char* fn) {
    const int nb = (int)(K / QK);
    CUtensorMap ta, tb;
    if (!make_map(&ta, xq, (uint64_t)nb * Q8_1_BYTES, (uint64_t)M, A_ROW, BM) ||
        !make_map(&tb, wq, (uint64_t)(FMT == FMT_Q8_0 ? nb * Q8_0_BYTES : nb / 8 * Q4_K_BYTES), (uint64_t)N,
                  b_row(FMT), BN)) {
        report(fn, MMQ_ERR_CUDA, "tensor map encoding failed");
        return MMQ_ERR_CUDA;
    }
    const int smem = Layout<FMT>::alloc;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(k_mmq_tc<FMT, DOTS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) {
            cudaGetLastError();
            report(fn, MMQ_ERR_SMEM, cudaGetErrorString(e));
            return MMQ_ERR_SMEM;
        }
        attr_done = true;
    }
    dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    k_mmq_tc<FMT, DOTS><<<grid, THREADS, smem, s>>>(ta, tb, (int)M, (int)N, nb, out, dots);
    return launch_status(fn);
}

}  // namespace

bool tc_available() { return true; }

int tc_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, int32_t* dots,
              cudaStream_t s) {
    const char* fn = fmt == FMT_Q8_0 ? (dots ? "mmq_debug_block_dots_q8_0" : "mmq_gemm_q8_0")
                                     : (dots ? "mmq_debug_block_dots_q4_k" : "mmq_gemm_q4_k");
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
