// Expert-grouped contraction (llama's mul_mat_id): activation row r is contracted with
// the weight matrix of expert row_expert[r] ("When Does a Kernel Win Surface?", sec.
// "Fused indexed-MoE prefill GEMM": the rows are counting-sorted by expert into tiles of
// at most 128 rows, and each tile stages one expert's weights once and amortizes them over
// all of that expert's rows in the tile).
//
// Everything runs on the device, in stream order, so the call is asynchronous and can be
// captured in a graph:
//   k_group_count    per-expert row counts (rows whose id is outside [0, E) are not counted);
//   k_group_plan     one CTA: exclusive scans of the counts and of the tiles per expert
//                    (ceil(count / 128)) -> row offsets of each expert in the sorted order,
//                    the tile list (first sorted row, expert) and its length;
//   k_group_scatter  one warp per row: takes the next sorted slot of its expert, records the
//                    original row for the store, copies the q8_1 row there; rows with an
//                    out-of-range id get an all-zero output row instead;
// then the tensor-core contraction over the tile list (gemm_tc.cu, GROUPED), which stores
// each sorted row to its original row.  The order of rows within an expert depends on the
// atomics, but every row's result is computed by the same arithmetic wherever it lands, so
// the output does not depend on it.
#include "common.cuh"

namespace mmq {
namespace {

constexpr int GT = 128;          // rows per tile (the contraction's BM)
constexpr int PLAN_THREADS = 1024;

__global__ void k_group_count(const int32_t* __restrict__ row_expert, int R, int E, int* __restrict__ counts) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < R; r += gridDim.x * blockDim.x) {
        const int e = row_expert[r];
        if (e >= 0 && e < E) atomicAdd(&counts[e], 1);
    }
}

__global__ void __launch_bounds__(PLAN_THREADS)
k_group_plan(const int* __restrict__ counts, int E, int* __restrict__ offsets, int* __restrict__ cursor,
             int2* __restrict__ tiles, int* __restrict__ ntiles) {
    __shared__ int s_rows[PLAN_THREADS], s_tiles[PLAN_THREADS];
    __shared__ int carry_rows, carry_tiles;
    const int t = threadIdx.x;
    if (t == 0) carry_rows = carry_tiles = 0;
    __syncthreads();
    for (int base = 0; base < E; base += PLAN_THREADS) {
        const int e = base + t;
        const int c = e < E ? counts[e] : 0;
        const int nt = (c + GT - 1) / GT;
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
            for (int j = 0; j < nt; ++j) tiles[tile0 + j] = make_int2(row0 + GT * j, e);
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

__global__ void k_group_scatter(const uint8_t* __restrict__ xq, const int32_t* __restrict__ row_expert, int R, int E,
                                int row16, int N, int* __restrict__ cursor, int* __restrict__ perm,
                                uint8_t* __restrict__ xs, float* __restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < R; r += warps) {
        const int e = row_expert[r];
        if (e < 0 || e >= E) {  // no expert: an all-zero output row
            for (int n = lane; n < N; n += 32) out[(long long)r * N + n] = 0.f;
            continue;
        }
        int pos = 0;
        if (lane == 0) {
            pos = atomicAdd(&cursor[e], 1);
            perm[pos] = r;
        }
        pos = __shfl_sync(0xffffffffu, pos, 0);
        const uint4* src = reinterpret_cast<const uint4*>(xq) + (long long)r * row16;
        uint4* dst = reinterpret_cast<uint4*>(xs) + (long long)pos * row16;
        for (int i = lane; i < row16; i += 32) dst[i] = __ldg(src + i);
    }
}

}  // namespace

int grouped_launch(int fmt, const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                   int64_t K, float* out, cudaStream_t s) {
    const char* fn = fmt == FMT_Q8_0   ? "mmq_gemm_grouped_q8_0"
                     : fmt == FMT_Q5_K ? "mmq_gemm_grouped_q5_k" : "mmq_gemm_grouped_q4_k";
    const int64_t nb = K / QK, row_bytes = nb * Q8_1_BYTES;
    const int64_t max_tiles = (R + GT - 1) / GT + (E < R ? E : R);  // each expert adds at most one partial tile
    if (max_tiles > 65535) {
        report(fn, MMQ_ERR_SHAPE, "too many row tiles for the grid (R / 128 + min(E, R) > 65535)");
        return MMQ_ERR_SHAPE;
    }
    // scratch: counts[E], offsets[E + 1], cursor[E], ntiles, tiles[max_tiles], perm[R], xs[R][row_bytes]
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t b_counts = up((size_t)E * 4), b_offsets = up((size_t)(E + 1) * 4), b_cursor = up((size_t)E * 4),
                 b_ntiles = 256, b_tiles = up((size_t)max_tiles * 8), b_perm = up((size_t)R * 4),
                 b_xs = up((size_t)R * row_bytes);
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
    uint8_t* xs = p + b_perm;
    if (cudaMemsetAsync(counts, 0, (size_t)E * 4, s) != cudaSuccess) {
        cudaGetLastError();
        scratch_free(ws, s);
        report(fn, MMQ_ERR_CUDA, "cudaMemsetAsync failed");
        return MMQ_ERR_CUDA;
    }
    const int cgrid = (int)((R + 255) / 256 < 1184 ? (R + 255) / 256 : 1184);
    {
        ProfScope ps("k_group_count", s);
        k_group_count<<<cgrid, 256, 0, s>>>(row_expert, (int)R, (int)E, counts);
    }
    {
        ProfScope ps("k_group_plan", s);
        k_group_plan<<<1, PLAN_THREADS, 0, s>>>(counts, (int)E, offsets, cursor, tiles, ntiles);
    }
    {
        ProfScope ps("k_group_scatter", s);
        const int sgrid = (int)((R + 7) / 8 < 1184 ? (R + 7) / 8 : 1184);
        k_group_scatter<<<sgrid, 256, 0, s>>>(static_cast<const uint8_t*>(xq), row_expert, (int)R, (int)E,
                                              (int)(row_bytes / 16), (int)N, cursor, perm, xs, out);
    }
    st = launch_status(fn);
    if (st == MMQ_OK)
        st = tc_grouped_launch(fmt, xs, wq, R, E, N, K, tiles, ntiles, max_tiles, offsets + 1, perm, out, s);
    scratch_free(ws, s);  // stream-ordered: after the kernels above
    return st;
}

}  // namespace mmq
