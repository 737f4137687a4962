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
// Warp roles (one 128 x 128 output tile per CTA, 448 threads):
//   warp 0     TMA producer: raw q8_1 rows (288 B per 256 values) and raw weight rows
//              (Q8_0: 272 B, Q4_K: one 144 B super-block) for a 256-value k-tile, as
//              2-D tensor copies into a 2-stage ring ("13 . r7-r8 raw-byte MMQ
//              kernel", sec. 2: shared memory holds raw quant bytes; sec. 3.1: whole
//              super-blocks, out-of-range rows zero-filled by the copy engine).
//   warp 1     TMEM owner and MMA issuer: per 32-block, two K=16 MMAs (M=128, N=128)
//              into one of four TMEM accumulators, then tcgen05.commit.
//   warps 2-5  converters: codes -> fp16 (sign-biased byte permute + one half2
//              subtract, exact) into the canonical K-major no-swizzle UMMA layout, and
//              the per-row / per-column block scales into a small scale ring
//              (Q4_K: d*sc_j and dmin*m_j from the 12 packed bytes, computed once per
//              (row, block) instead of per lane, as in sec. 3.2 of the same page).
//   warps 6-13 epilogue: per 32-block, tcgen05.ld of the f32 block dots, then
//              acc += (xd*wd) * D (Q4_K: wd = d*sc_j, and acc -= dmin*m_j*xs) in f32
//              registers; at the end the tile is stored to out.
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
constexpr int FS = 4;                   // fp16 operand / scale slots (one 32-block each)
constexpr int DS = 4;                   // TMEM accumulators (one 32-block each)
constexpr int CONV_WARPS = 4;
constexpr int EPI_WARPS = 8;
constexpr int WARP_TMA = 0, WARP_MMA = 1, WARP_CONV0 = 2, WARP_EPI0 = WARP_CONV0 + CONV_WARPS;
constexpr int THREADS = (WARP_EPI0 + EPI_WARPS) * 32;
constexpr int TMEM_COLS = DS * BN;      // 512: the whole TMEM of the SM
constexpr int A_ROW = KT_BLOCKS * Q8_1_BYTES;  // 288
constexpr int OP_A = BM * QK * 2;       // fp16 A tile of one block: 8 KiB
constexpr int OP_B = BN * QK * 2;       // fp16 B tile of one block: 8 KiB
constexpr int SC_FLOATS = 2 * BM + 2 * BN;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

static_assert(BM == 32 * CONV_WARPS && BN == 32 * CONV_WARPS, "one scale row per converter thread");
static_assert(EPI_WARPS == 8 && BN == 128, "epilogue covers 4 lane quarters x 2 column halves of 64");

__host__ __device__ constexpr int b_row(int fmt) { return fmt == FMT_Q8_0 ? KT_BLOCKS * Q8_0_BYTES : Q4_K_BYTES; }

// barrier indices.  One slot holds the fp16 operands and the scales of one 32-block:
// SLOT_FULL is arrived by every converter warp; SLOT_EMPTY by the MMA commit (operands
// read) and by every epilogue warp (scales read).
constexpr int BAR_RAW_FULL = 0, BAR_RAW_EMPTY = BAR_RAW_FULL + RS, BAR_SLOT_FULL = BAR_RAW_EMPTY + RS,
              BAR_SLOT_EMPTY = BAR_SLOT_FULL + FS, BAR_D_FULL = BAR_SLOT_EMPTY + FS, BAR_D_EMPTY = BAR_D_FULL + DS,
              BAR_DRAIN = BAR_D_EMPTY + DS, NBARS = BAR_DRAIN + 1;

template <int FMT>
struct Layout {
    static constexpr int rawA = 0;
    static constexpr int rawB = rawA + RS * BM * A_ROW;
    static constexpr int opA = rawB + RS * BN * b_row(FMT);
    static constexpr int opB = opA + FS * OP_A;
    static constexpr int sc = opB + FS * OP_B;
    static constexpr int bars = sc + FS * SC_FLOATS * 4;
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
    for (uint32_t i = 1;; ++i) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 0) {
            if (*abort) return false;
            if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                atomicOr(&g_tc_error, ERR_TIMEOUT);
                *abort = 1;
                return false;
            }
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

// Every lane polls the same phase; the vote keeps the warp on one path (a phase that
// one lane saw complete cannot be reused before this warp arrives on its partner).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const bool ok = wait_bar(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
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
        for (int s = 0; s < RS; ++s) {
            ptx::mbar_init(bar(BAR_RAW_FULL + s), 1);
            ptx::mbar_init(bar(BAR_RAW_EMPTY + s), CONV_WARPS);
        }
        for (int f = 0; f < FS; ++f) {
            ptx::mbar_init(bar(BAR_SLOT_FULL + f), CONV_WARPS);
            ptx::mbar_init(bar(BAR_SLOT_EMPTY + f), 1 + EPI_WARPS);
        }
        for (int t = 0; t < DS; ++t) {
            ptx::mbar_init(bar(BAR_D_FULL + t), 1);
            ptx::mbar_init(bar(BAR_D_EMPTY + t), EPI_WARPS);
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
            for (int bi = 0; bi < nb; ++bi) {
                const int f = bi % FS, t = bi % DS;
                if (!wait_bar(bar(BAR_SLOT_FULL + f), (bi / FS) & 1, abort)) break;
                if (!wait_bar(bar(BAR_D_EMPTY + t), ((bi / DS) & 1) ^ 1, abort)) break;
                ptx::tc_fence_after();
                const uint32_t a = sbase + L::opA + f * OP_A, b = sbase + L::opB + f * OP_B;
                const uint32_t d = tmem + (uint32_t)(t * BN);
                ptx::umma_f16(d, sdesc(a), sdesc(b), idesc, 0u);
                ptx::umma_f16(d, sdesc(a + 256), sdesc(b + 256), idesc, 1u);
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
        const int ct = cw * 32 + lane;
        const int r8 = lane & 7, half = (lane >> 3) & 1, kgl = lane >> 4;
        bool ok = true;
        for (int kt = 0; kt < nkt && ok; ++kt) {
            const int s = kt % RS;
            ok = warp_wait(bar(BAR_RAW_FULL + s), (kt / RS) & 1, abort);
            if (!ok) break;
            const uint8_t* rA = smem + L::rawA + s * BM * A_ROW;
            const uint8_t* rB = smem + L::rawB + s * BN * BROW;
            for (int j = 0; j < KT_BLOCKS; ++j) {
                const int bi = kt * KT_BLOCKS + j, f = bi % FS;
                ok = warp_wait(bar(BAR_SLOT_EMPTY + f), ((bi / FS) & 1) ^ 1, abort);
                if (!ok) break;
                uint8_t* oA = smem + L::opA + f * OP_A;
                uint8_t* oB = smem + L::opB + f * OP_B;
                float* sc = reinterpret_cast<float*>(smem + L::sc + f * SC_FLOATS * 4);
                // All raw loads first (the stores below go to the same shared array, so
                // the compiler would otherwise keep every load behind the previous store).
                // Unit i: 8-row group g and a pair of 8-value k-groups; each lane takes
                // one 4-code word = half of one core-matrix row.
                uint32_t xa[8], wv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int u = i * CONV_WARPS + cw;
                    const int g = u >> 1, kg = (u & 1) * 2 + kgl, w = kg * 2 + half, r = g * 8 + r8;
                    xa[i] = *reinterpret_cast<const uint32_t*>(rA + r * A_ROW + j * Q8_1_BYTES + 4 + w * 4);
                    if (FMT == FMT_Q8_0) {
                        // codes start at an odd half-word for even j: two aligned words
                        // and a funnel shift (for odd j the second load is the first)
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
                const uint32_t hd = *reinterpret_cast<const uint32_t*>(rA + ct * A_ROW + j * Q8_1_BYTES);
                float wsc, wmn;
                if (FMT == FMT_Q8_0) {
                    wsc = f16_bits_to_f32(*reinterpret_cast<const unsigned short*>(rB + ct * BROW + j * Q8_0_BYTES));
                    wmn = 0.f;
                } else {
                    const uint4 p = *reinterpret_cast<const uint4*>(rB + ct * BROW);
                    int s6, m6;
                    q4_k_scale_min(p.y, p.z, p.w, j, s6, m6);
                    wsc = f16_bits_to_f32(p.x) * (float)s6;        // exact
                    wmn = f16_bits_to_f32(p.x >> 16) * (float)m6;  // exact
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int u = i * CONV_WARPS + cw;
                    const int g = u >> 1, kg = (u & 1) * 2 + kgl;
                    const int dst = g * 512 + kg * 128 + r8 * 16 + half * 8;
                    *reinterpret_cast<uint2*>(oA + dst) = i8x4_to_f16x4(xa[i]);
                    *reinterpret_cast<uint2*>(oB + dst) =
                        FMT == FMT_Q8_0 ? i8x4_to_f16x4(wv[i]) : u4x4_to_f16x4(wv[i]);
                }
                sc[ct] = f16_bits_to_f32(hd);
                sc[BM + ct] = f16_bits_to_f32(hd >> 16);
                sc[2 * BM + ct] = wsc;
                sc[2 * BM + BN + ct] = wmn;
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BAR_SLOT_FULL + f));
            }
            __syncwarp();
            if (ok && lane == 0) ptx::mbar_arrive(bar(BAR_RAW_EMPTY + s));
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                    // TMEM lane quarter this warp may access
        const int h = (warp - WARP_EPI0) >> 2;     // column half
        const int mloc = 32 * q + lane;
        const int mrow = m0 + mloc;
        float acc[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) acc[c] = 0.f;
        for (int bi = 0; bi < nb; ++bi) {
            const int t = bi % DS, f = bi % FS;
            if (!(warp_wait(bar(BAR_D_FULL + t), (bi / DS) & 1, abort) &&
                  warp_wait(bar(BAR_SLOT_FULL + f), (bi / FS) & 1, abort)))
                break;
            ptx::tc_fence_after();
            const float* sc = reinterpret_cast<const float*>(smem + L::sc + f * SC_FLOATS * 4);
            const float xd = sc[mloc];
            const float nxs = -sc[BM + mloc];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t dv[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(t * BN + 64 * h + 32 * c2), dv);
                ptx::tmem_ld_wait(dv);
                const int col0 = 64 * h + 32 * c2;
                if (DOTS) {
                    if (mrow < M) {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int n = n0 + col0 + c;
                            if (n < N)
                                dots[((long long)mrow * N + n) * nb + bi] = __float2int_rn(__uint_as_float(dv[c]));
                        }
                    }
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 w = *reinterpret_cast<const float4*>(sc + 2 * BM + col0 + 4 * c4);
                        const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = 4 * c4 + e;
                            acc[32 * c2 + c] = fmaf(xd * wv[e], __uint_as_float(dv[c]), acc[32 * c2 + c]);
                        }
                        if (FMT == FMT_Q4_K) {
                            const float4 mn = *reinterpret_cast<const float4*>(sc + 2 * BM + BN + col0 + 4 * c4);
                            const float mv[4] = {mn.x, mn.y, mn.z, mn.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                acc[32 * c2 + 4 * c4 + e] = fmaf(mv[e], nxs, acc[32 * c2 + 4 * c4 + e]);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(bar(BAR_D_EMPTY + t));
                ptx::mbar_arrive(bar(BAR_SLOT_EMPTY + f));
            }
        }
        if (!DOTS && mrow < M && !*abort) {
            float* orow = out + (long long)mrow * N + n0 + 64 * h;
            const int ncols = min(64, N - (n0 + 64 * h));
            if (ncols == 64 && (N & 3) == 0) {
#pragma unroll
                for (int c = 0; c < 64; c += 4)
                    *reinterpret_cast<float4*>(orow + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                    if (c < ncols) orow[c] = acc[c];
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
