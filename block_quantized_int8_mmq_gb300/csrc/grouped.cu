// Expert-grouped contraction (llama's mul_mat_id): activation row r is contracted with
// the weight matrix of expert row_expert[r] ("When Does a Kernel Win Surface?", sec.
// "Fused indexed-MoE prefill GEMM": the rows are counting-sorted by expert into tiles of
// at most 128 rows, and each tile stages one expert's weights once and amortizes them over
// all of that expert's rows in the tile).
//
// Everything runs on the device, in stream order, so the call is asynchronous and can be
// captured in a graph:
//   k_group_count    per-expert row counts (rows whose id is outside [0, E) are not counted):
//                    per-CTA histograms in shared memory, one global add per CTA and expert;
//   k_group_plan     one CTA (which also counts the ids itself, in shared memory, for up to
//                    PLAN_COUNT_ROWS rows and SMEM_EXPERTS experts: then no k_group_count and
//                    no clearing of the counts): exclusive scans of the counts and of the tiles per expert
//                    (ceil(count / 128)) -> row offsets of each expert in the sorted order,
//                    the tile list (first sorted row, expert) and its length;
//   k_group_scatter  a CTA per 256 rows: ranks its rows within each expert in shared
//                    memory, reserves one range of sorted slots per expert (a global add on
//                    the expert's cursor) and records each row's original index at its slot;
//                    rows with an out-of-range id get an all-zero output row instead;
//   k_group_copy     (the converter kernel only) one warp per sorted slot: the q8_1 row
//                    copied there;
// then a contraction over the tile list, which stores each sorted row to its original row:
// the converter kernel (gemm_tc.cu, GROUPED) on the sorted copy, the expanded path
// (gemm_expand.cu), whose expansion gathers each tile's rows from xq through the
// permutation and expands the weights of every expert that has rows, or, for experts with
// few rows, the dp4a weight stream (gemm_small.cu, GROUPED) over tiles of 2 or 4 rows: the
// tile height follows the experts' fill ("Fused indexed-MoE prefill GEMM", dynamic M-tile),
// 128-row tensor-core tiles where experts have many rows, weight-streaming tiles where a
// 128-row tile would be almost empty.  The order of rows within an expert depends on the
// atomics, but every row's result is computed by the same arithmetic wherever it lands, so
// the output does not depend on it.
#include "common.cuh"

namespace mmq {
namespace {

constexpr int GT = 128;          // rows per tile of the tensor-core contractions (their BM)
constexpr int PLAN_THREADS = 1024;
constexpr int SMEM_EXPERTS = 8192;  // per-expert counters in shared memory up to this many experts
constexpr int GROUP_THREADS = 256;  // rows per counting / ranking CTA (one per thread)

// Per-CTA counts in shared memory (E <= SMEM_EXPERTS), else global adds per row.
__global__ void __launch_bounds__(GROUP_THREADS)
k_group_count(const int32_t* __restrict__ row_expert, int R, int E, int* __restrict__ counts) {
    extern __shared__ int hist[];
    const bool local = E <= SMEM_EXPERTS;
    if (local) {
        for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
        __syncthreads();
    }
    const int r = blockIdx.x * GROUP_THREADS + threadIdx.x;
    const int e = r < R ? row_expert[r] : -1;
    if (e >= 0 && e < E) atomicAdd(local ? &hist[e] : &counts[e], 1);
    if (local) {
        __syncthreads();
        for (int i = threadIdx.x; i < E; i += blockDim.x)
            if (hist[i]) atomicAdd(&counts[i], hist[i]);
    }
}

constexpr int PLAN_COUNT_ROWS = 65536;

// counts == nullptr: the CTA counts the R ids of row_expert itself (E <= SMEM_EXPERTS)
__global__ void __launch_bounds__(PLAN_THREADS)
k_group_plan(const int32_t* __restrict__ row_expert, int R, const int* __restrict__ counts, int E, int gt,
             int* __restrict__ offsets, int* __restrict__ cursor, int2* __restrict__ tiles, int* __restrict__ ntiles) {
    extern __shared__ int hist[];
    __shared__ int s_rows[PLAN_THREADS], s_tiles[PLAN_THREADS];
    __shared__ int carry_rows, carry_tiles;
    const int t = threadIdx.x;
    if (t == 0) carry_rows = carry_tiles = 0;
    if (!counts) {
        for (int i = t; i < E; i += PLAN_THREADS) hist[i] = 0;
        __syncthreads();
        // eight ids per thread loaded before their adds (one memory round trip per batch)
        constexpr int B = 8;
        for (int r0 = 0; r0 < R; r0 += B * PLAN_THREADS) {
            int ids[B];
#pragma unroll
            for (int u = 0; u < B; ++u) {
                const int r = r0 + u * PLAN_THREADS + t;
                ids[u] = r < R ? row_expert[r] : -1;
            }
#pragma unroll
            for (int u = 0; u < B; ++u)
                if (ids[u] >= 0 && ids[u] < E) atomicAdd(&hist[ids[u]], 1);
        }
    }
    __syncthreads();
    for (int base = 0; base < E; base += PLAN_THREADS) {
        const int e = base + t;
        const int c = e < E ? (counts ? counts[e] : hist[e]) : 0;
        const int nt = (c + gt - 1) / gt;
        s_rows[t] = c;
        s_tiles[t] = nt;
        __syncthreads();
        for (int off = 1; off < PLAN_THREADS; off <<= 1) {  // inclusive scans (Hillis-Steele)
            const int a = t >= off ? s_rows[t - off] : 0, b = t >= off ? s_tiles[t - off] : 0;
            __syncthreads();
            s_rows[t] += a;
            s_tiles[t] += b;
            __syncthreads();
        }
        const int row0 = carry_rows + s_rows[t] - c, tile0 = carry_tiles + s_tiles[t] - nt;
        if (e < E) {
            offsets[e] = row0;
            cursor[e] = row0;
            for (int j = 0; j < nt; ++j) tiles[tile0 + j] = make_int2(row0 + gt * j, e);
        }
        __syncthreads();
        if (t == PLAN_THREADS - 1) {
            carry_rows += s_rows[t];
            carry_tiles += s_tiles[t];
        }
        __syncthreads();
    }
    if (t == 0) {
        offsets[E] = carry_rows;
        *ntiles = carry_tiles;
    }
}

// CTA c takes rows 256c .. 256c + 255; with E <= SMEM_EXPERTS it ranks them per expert in
// shared memory and reserves one range of slots per expert, else one global add per row.
__global__ void __launch_bounds__(GROUP_THREADS)
k_group_scatter(const int32_t* __restrict__ row_expert, int R, int E, int N, int* __restrict__ cursor,
                int* __restrict__ perm, float* __restrict__ out) {
    extern __shared__ int hist[];  // E counters
    const bool local = E <= SMEM_EXPERTS;
    if (local) {
        for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
        __syncthreads();
    }
    const int r = blockIdx.x * GROUP_THREADS + threadIdx.x;
    const int e = r < R ? row_expert[r] : -1;
    const bool valid = e >= 0 && e < E;
    // the row's rank within its expert in this CTA (or, without the shared counters, its slot)
    const int rank = !valid ? -1 : local ? atomicAdd(&hist[e], 1) : atomicAdd(&cursor[e], 1);
    if (local) {
        __syncthreads();
        // one range of slots per expert with rows here: hist[e] becomes its first slot
        for (int i = threadIdx.x; i < E; i += blockDim.x)
            if (hist[i]) hist[i] = atomicAdd(&cursor[i], hist[i]);
        __syncthreads();
    }
    if (valid) perm[local ? hist[e] + rank : rank] = r;
    // an out-of-range id: an all-zero output row (the warp's such rows, one after another)
    const int lane = threadIdx.x & 31;
    unsigned bad = __ballot_sync(0xffffffffu, r < R && !valid);
    while (bad) {
        const int i = __ffs(bad) - 1;
        bad &= bad - 1;
        const long long row = (long long)(r - lane + i);
        for (int n = lane; n < N; n += 32) out[row * N + n] = 0.f;
    }
}

// The converter kernel's input: sorted row p (p < rows) is q8_1 row perm[p] of xq.
__global__ void k_group_copy(const uint8_t* __restrict__ xq, const int* __restrict__ perm, const int* __restrict__ rows,
                             int R, int row16, uint8_t* __restrict__ xs) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5), n = min(R, *rows);
    for (int p = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < n; p += warps) {
        const uint4* src = reinterpret_cast<const uint4*>(xq) + (long long)perm[p] * row16;
        uint4* dst = reinterpret_cast<uint4*>(xs) + (long long)p * row16;
        for (int i = lane; i < row16; i += 32) dst[i] = __ldg(src + i);
    }
}

}  // namespace

// the grouped dp4a stream (gemm_small.cu)
bool small_grouped_fits(int fmt, int64_t K, int mt);
int small_grouped_launch(int fmt, const void* xq, const void* wq, int64_t R, int64_t E, int64_t N, int64_t K,
                         const int2* tiles, const int* ntiles, int64_t max_tiles, const int* offsets, const int* perm,
                         int mt, float* out, cudaStream_t s, const char* fn);

// Average rows per expert up to which MMQ_PATH_AUTO takes the grouped weight stream: it reads
// an expert's weights once per tile of 2 or 4 rows, the expanded path writes and reads every
// expert's expanded weights once.  Measured on 128 experts of 768 x 2048 (stream / expanded,
// us): Q4_K 1 row per expert 48 / 166, 4 rows 126 / 255, 8 rows 218 / 257, 16 rows 377 /
// 259; Q5_K 8 rows 229 / 261, 10 rows 264 / 261; Q6_K 1 row 62 / 233, 8 rows 357 / 353;
// Q8_0 8 rows 165 / 249, 12 rows 220 / 250.
static int64_t stream_rows_per_expert(int fmt) {
    return fmt == FMT_Q8_0 ? 14 : fmt == FMT_Q4_K ? 10 : fmt == FMT_Q5_K ? 9 : 7;
}

// path: MMQ_PATH_TC (the converter kernel), MMQ_PATH_EXPAND, MMQ_PATH_SMALL (the grouped
// weight stream) or MMQ_PATH_AUTO (the stream for up to stream_rows_per_expert rows per
// expert on average, else the expanded path); *taken: the contraction used
int grouped_launch_path(int fmt, const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E,
                        int64_t N, int64_t K, float* out, cudaStream_t s, int path, int* taken) {
    const char* fn = fmt == FMT_Q8_0   ? "mmq_gemm_grouped_q8_0"
                     : fmt == FMT_Q5_K ? "mmq_gemm_grouped_q5_k"
                     : fmt == FMT_Q6_K ? "mmq_gemm_grouped_q6_k" : "mmq_gemm_grouped_q4_k";
    const bool use_tc = path == MMQ_PATH_TC;
    // the stream's tile height: 2 rows where experts hold about one row, else 4
    const int mt = R <= 2 * E ? 2 : 4;
    bool stream = path == MMQ_PATH_SMALL || (path == MMQ_PATH_AUTO && R <= stream_rows_per_expert(fmt) * E);
    if (stream && !small_grouped_fits(fmt, K, mt)) {
        if (path == MMQ_PATH_SMALL) {
            report(fn, MMQ_ERR_SHAPE, "K too large for the grouped weight stream's shared memory");
            return MMQ_ERR_SHAPE;
        }
        stream = false;
    }
    const int gt = stream ? mt : GT;
    const int64_t nb = K / QK, row_bytes = nb * Q8_1_BYTES;
    const int64_t max_tiles = (R + gt - 1) / gt + (E < R ? E : R);  // each expert adds at most one partial tile
    if (max_tiles > 65535) {
        report(fn, MMQ_ERR_SHAPE, stream ? "too many row tiles for the grid (R / tile rows + min(E, R) > 65535)"
                                         : "too many row tiles for the grid (R / 128 + min(E, R) > 65535)");
        return MMQ_ERR_SHAPE;
    }
    // scratch: counts[E], offsets[E + 1], cursor[E], ntiles, tiles[max_tiles], perm[R], and for
    // the converter kernel xs[R][row_bytes]
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t b_counts = up((size_t)E * 4), b_offsets = up((size_t)(E + 1) * 4), b_cursor = up((size_t)E * 4),
                 b_ntiles = 256, b_tiles = up((size_t)max_tiles * 8), b_perm = up((size_t)R * 4),
                 b_xs = use_tc ? up((size_t)R * row_bytes) : 0;
    void* ws = nullptr;
    int st = scratch_alloc(b_counts + b_offsets + b_cursor + b_ntiles + b_tiles + b_perm + b_xs, s, &ws, fn);
    if (st != MMQ_OK) return st;
    uint8_t* p = static_cast<uint8_t*>(ws);
    int* counts = reinterpret_cast<int*>(p);
    int* offsets = reinterpret_cast<int*>(p += b_counts);
    int* cursor = reinterpret_cast<int*>(p += b_offsets);
    int* ntiles = reinterpret_cast<int*>(p += b_cursor);
    int2* tiles = reinterpret_cast<int2*>(p += b_ntiles);
    int* perm = reinterpret_cast<int*>(p += b_tiles);
    uint8_t* xs = use_tc ? p + b_perm : nullptr;
    const size_t hist_bytes = E <= SMEM_EXPERTS ? (size_t)E * 4 : 0;
    const unsigned rgrid = (unsigned)((R + GROUP_THREADS - 1) / GROUP_THREADS);
    const bool count_in_plan = R <= PLAN_COUNT_ROWS && E <= SMEM_EXPERTS;
    if (!count_in_plan) {
        if (cudaMemsetAsync(counts, 0, (size_t)E * 4, s) != cudaSuccess) {
            cudaGetLastError();
            scratch_free(ws, s);
            report(fn, MMQ_ERR_CUDA, "cudaMemsetAsync failed");
            return MMQ_ERR_CUDA;
        }
        ProfScope ps("k_group_count", s);
        k_group_count<<<rgrid, GROUP_THREADS, hist_bytes, s>>>(row_expert, (int)R, (int)E, counts);
    }
    {
        ProfScope ps("k_group_plan", s);
        k_group_plan<<<1, PLAN_THREADS, count_in_plan ? hist_bytes : 0, s>>>(
            row_expert, (int)R, count_in_plan ? nullptr : counts, (int)E, gt, offsets, cursor, tiles, ntiles);
    }
    {
        ProfScope ps("k_group_scatter", s);
        k_group_scatter<<<rgrid, GROUP_THREADS, hist_bytes, s>>>(row_expert, (int)R, (int)E, (int)N, cursor, perm,
                                                                 out);
    }
    if (use_tc) {
        ProfScope ps("k_group_copy", s);
        const int64_t cg = (R + 7) / 8;
        k_group_copy<<<(unsigned)(cg < 4736 ? cg : 4736), 256, 0, s>>>(static_cast<const uint8_t*>(xq), perm,
                                                                       offsets + E, (int)R, (int)(row_bytes / 16), xs);
    }
    st = launch_status(fn);
    if (st == MMQ_OK && stream)
        st = small_grouped_launch(fmt, xq, wq, R, E, N, K, tiles, ntiles, max_tiles, offsets, perm, mt, out, s, fn);
    else if (st == MMQ_OK && use_tc)
        st = tc_grouped_launch(fmt, xs, wq, R, E, N, K, tiles, ntiles, max_tiles, offsets + 1, perm, out, s);
    else if (st == MMQ_OK)
        st = tcx_grouped_launch(fmt, xq, R, wq, E, N, K, tiles, ntiles, max_tiles, offsets, perm, out, s, fn);
    scratch_free(ws, s);  // stream-ordered: after the kernels above
    if (st == MMQ_OK && taken) *taken = stream ? MMQ_PATH_SMALL : use_tc ? MMQ_PATH_TC : MMQ_PATH_EXPAND;
    return st;
}

int grouped_launch(int fmt, const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                   int64_t K, float* out, cudaStream_t s, bool use_tc) {
    return grouped_launch_path(fmt, xq, row_expert, R, wq, E, N, K, out, s, use_tc ? MMQ_PATH_TC : MMQ_PATH_EXPAND,
                               nullptr);
}

}  // namespace mmq
