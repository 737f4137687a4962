// C ABI of libmmq: argument checks, kernel selection and the error protocol.
//
// Error protocol ("13 . r7-r8 raw-byte MMQ kernel", sec. 3.3, the silent-failure
// lesson): every call returns a status; a refused call launches nothing and prints one
// stderr line; a failed launch is read with cudaGetLastError (which also clears it) and
// reported, so a benchmark can never time a kernel that did not run.
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "common.cuh"

namespace mmq {

void report(const char* fn, int status, const char* detail) {
    fprintf(stderr, "libmmq: %s refused: %s (%s)\n", fn, mmq_status_string(status), detail);
}

int launch_status(const char* fn) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        fprintf(stderr, "libmmq: %s launch failed: %s\n", fn, cudaGetErrorString(e));
        return MMQ_ERR_LAUNCH;
    }
    return MMQ_OK;
}

bool tc_available();

DeviceShape device_shape() {
    static std::atomic<int> sms[MAX_DEVICES], smem[MAX_DEVICES], l2[MAX_DEVICES];
    const DeviceShape fallback{152, 233472, 132 << 20};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return fallback;
    }
    if (sms[dev].load() == 0) {
        int a = 0, b = 0, c = 0;
        if (cudaDeviceGetAttribute(&a, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&b, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&c, cudaDevAttrL2CacheSize, dev) != cudaSuccess || a <= 0) {
            cudaGetLastError();
            return fallback;
        }
        smem[dev].store(b);
        l2[dev].store(c);
        sms[dev].store(a);
    }
    DeviceShape d;
    d.sms = sms[dev].load();
    d.smem_per_sm = smem[dev].load();
    d.l2_bytes = l2[dev].load();
    return d;
}

namespace {
std::atomic<int> g_refuse_smem{0};  // test switch: every shared-memory request is refused
}  // namespace

int ensure_smem(const void* func, int bytes, SmemAttr& a) {
    if (g_refuse_smem.load()) return MMQ_ERR_SMEM;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    if (a.bytes[dev].load() >= bytes) return MMQ_OK;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_SMEM;
    }
    int cur = a.bytes[dev].load();
    while (cur < bytes && !a.bytes[dev].compare_exchange_weak(cur, bytes)) {
    }
    return MMQ_OK;
}

// The expert-grouped call on the contraction `path` names (MMQ_PATH_AUTO: by the experts'
// average fill); *taken: the one used (grouped.cu).
int grouped_launch_path(int fmt, const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E,
                        int64_t N, int64_t K, float* out, cudaStream_t s, int path, int* taken);

// Time of the Q6_K tensor-core stream for M x N x K (us, measured on GB300: per wave of
// CTAs, one per SM, ~1.9 us per two-super-block chunk of a CTA's share of K, plus ~3.5 us
// until the first chunk is in), or -1 where the stream does not take the shape (gemm_small.cu).
double q6_stream_cost_us(int64_t M, int64_t N, int64_t K);

// Test switch of the Q8_0 / Q4_K / Q5_K tensor-core streams' K splits (0: the measured rule,
// n > 0: n splits) and boxes per CTA with a forced split (0: the launcher's) (gemm_small.cu).
void small_set_ksplit(int splits, int boxes);
// The Q8_0 / Q4_K / Q5_K tensor-core stream's grid for a shape under stream capture: boxes
// per CTA and K splits (gemm_small.cu; host only).
void small_stream_grid(int fmt, int64_t M, int64_t N, int64_t K, int32_t* boxes, int32_t* splits);

namespace {

std::atomic<int> g_path{-1};
thread_local int t_last_path = 0;

int current_path() {
    int p = g_path.load();
    if (p < 0) {
        p = MMQ_PATH_AUTO;
        const char* env = getenv("MMQ_FORCE_PATH");
        if (env && strcmp(env, "small") == 0) p = MMQ_PATH_SMALL;
        if (env && strcmp(env, "tc") == 0) p = MMQ_PATH_TC;
        if (env && strcmp(env, "expand") == 0) p = MMQ_PATH_EXPAND;
        int expected = -1;
        g_path.compare_exchange_strong(expected, p);
        p = g_path.load();
    }
    return p;
}

constexpr int64_t LIMIT = (int64_t)1 << 40;

// Path choice for MMQ_PATH_AUTO from two cost models fitted to measurements on GB300
// (microseconds, M from 8 to 384 on 512..18944 x 3584..18944 weights):
// - the small-M streams take the weights once per pass of 8 activation rows, at about 4.4
//   million weight values per microsecond, a quarter less when the weights are small (N * K
//   below 32 M values: too little work per pass to fill the GPU); Q6_K: its tensor-core
//   stream's own model (q6_stream_cost_us: waves of CTAs times chunks per CTA), or, for
//   the shapes that stream does not take, 4 rows per pass at 2.7 (0.82 of it when small);
// - the expanded tensor-core path pays the code expansion (~0.6 us per million weight
//   values; Q6_K, two planes: ~1.0) plus, per wave of output tiles (times their K splits)
//   over the SMs, one CTA's pass over its share of K (~0.28 us per 32-block of a 128-wide
//   tile; the K-quants with mins add one min item per 8 blocks), plus fixed costs.
// The converter kernel is never the faster of the two and is only used when asked for.
int auto_path(int fmt, int64_t M, int64_t N, int64_t K) {
    if (M <= 8 || K % QK_K != 0 || !tc_available()) return MMQ_PATH_SMALL;
    const bool q6 = fmt == FMT_Q6_K;
    const double nk = (double)N * (double)K;
    const double t_q6s = q6 ? q6_stream_cost_us(M, N, K) : -1.0;
    const double rate = (q6 ? 2.7e6 : 4.4e6) * (nk < 32e6 ? (q6 ? 0.82 : 0.77) : 1.0);
    const double t_small = t_q6s >= 0 ? t_q6s : (double)(q6 ? (M + 3) / 4 : (M + 7) / 8) * nk / rate + 1.5;
    // with K split S ways (small outputs), S times the CTAs each take 1/S of the groups,
    // and a summing kernel follows
    const int64_t S = tcx_splits(fmt, M, N, K), ng = K / QK_K, bn = tcx_tile_n(fmt, M, N), sms = device_shape().sms;
    const int64_t ctas = ((M + 127) / 128) * ((N + bn - 1) / bn) * S;
    const double waves = (double)((ctas + sms - 1) / sms);
    const double items = (double)(8 * ((ng + S - 1) / S)) * (is_kquant(fmt) ? 9.0 / 8.0 : 1.0) * (double)bn / 128.0;
    const double t_expand =
        (q6 ? 1.0 : 0.6) * nk / 1e6 + 0.28 * waves * items + (q6 ? 5.0 : 8.0) + (S > 1 ? 1.0 : 0.0);
    return t_small < t_expand ? MMQ_PATH_SMALL : MMQ_PATH_EXPAND;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_mk(const char* fn, int64_t M, int64_t N, int64_t K, int64_t kmul) {
    if (M < 1 || N < 1 || K < 1) {
        report(fn, MMQ_ERR_SHAPE, "M, N and K must be >= 1");
        return MMQ_ERR_SHAPE;
    }
    if (K % kmul != 0) {
        report(fn, MMQ_ERR_K_MULTIPLE, kmul == 256 ? "K % 256 != 0" : "K % 32 != 0");
        return MMQ_ERR_K_MULTIPLE;
    }
    if (M > LIMIT / K || N > LIMIT / K || M > LIMIT / N || K / QK > 0x7fffffff || N > 0x7fffffff ||
        M > 0x7fffffff) {
        report(fn, MMQ_ERR_SHAPE, "size product too large");
        return MMQ_ERR_SHAPE;
    }
    return MMQ_OK;
}

int contraction(const char* fn, int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K,
                float* out, int32_t* dots, void* stream) {
    int st = check_mk(fn, M, N, K, is_superblock(fmt) ? QK_K : QK);
    if (st) return st;
    void* o = out ? static_cast<void*>(out) : static_cast<void*>(dots);
    if (!xq || !wq || !o) {
        report(fn, MMQ_ERR_NULL, "xq, wq and the output must be non-NULL");
        return MMQ_ERR_NULL;
    }
    if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(o, 16)) {
        report(fn, MMQ_ERR_ALIGN, "xq, wq and the output must be 16-byte aligned");
        return MMQ_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int path = current_path();
    if (path == MMQ_PATH_AUTO) path = auto_path(fmt, M, N, K);
    if (path == MMQ_PATH_SMALL)
        st = small_launch(fmt, xq, wq, M, N, K, out, dots, s);
    else if (path == MMQ_PATH_TC)
        st = tc_launch(fmt, xq, wq, M, N, K, out, dots, s);
    else
        st = tcx_launch(fmt, xq, wq, M, N, K, out, dots, s, false);
    if (st == MMQ_OK) t_last_path = path;
    return st;
}

// Quantize + contraction in one call.  On the expanded-code path the quantization is
// fused into the activation expansion (one pass over x writes both xq and the fp16
// operand); on the other paths it is the quantize kernel followed by the contraction.
int linear(const char* fn, int fmt, const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq,
           float* out, void* stream) {
    int st = check_mk(fn, M, N, K, is_superblock(fmt) ? QK_K : QK);
    if (st) return st;
    if (!x || !xq || !wq || !out) {
        report(fn, MMQ_ERR_NULL, "x, xq, wq and out must be non-NULL");
        return MMQ_ERR_NULL;
    }
    if (!aligned(x, 16) || !aligned(xq, 16) || !aligned(wq, 16) || !aligned(out, 16)) {
        report(fn, MMQ_ERR_ALIGN, "x, xq, wq and out must be 16-byte aligned");
        return MMQ_ERR_ALIGN;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int path = current_path();
    if (path == MMQ_PATH_AUTO) path = auto_path(fmt, M, N, K);
    if (path == MMQ_PATH_EXPAND) {
        st = tcx_linear_launch(fmt, x, xq, wq, M, N, K, out, s);
    } else {
        st = quantize_launch(x, M, K, xq, s);
        if (st == MMQ_OK)
            st = path == MMQ_PATH_SMALL ? small_launch(fmt, xq, wq, M, N, K, out, nullptr, s)
                                        : tc_launch(fmt, xq, wq, M, N, K, out, nullptr, s);
    }
    if (st == MMQ_OK) t_last_path = path;
    return st;
}

// Expert-grouped contraction: rows grouped by expert on the device, then a tensor-core
// contraction over the tile list (needs tcgen05 and K % 256 == 0): the converter kernel
// when MMQ_PATH_TC is set (not Q6_K), else the expanded path.
int grouped(const char* fn, int fmt, const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E,
            int64_t N, int64_t K, float* out, void* stream) {
    int st = check_mk(fn, R, N, K, QK_K);
    if (st) return st;
    if (E < 1 || E > (int64_t)1 << 20 || E * N > 0x7fffffff || E > LIMIT / N / (K / QK)) {
        report(fn, MMQ_ERR_SHAPE, "E must be in 1 .. 2^20 and E*N rows below 2^31");
        return MMQ_ERR_SHAPE;
    }
    if (!xq || !row_expert || !wq || !out) {
        report(fn, MMQ_ERR_NULL, "xq, row_expert, wq and out must be non-NULL");
        return MMQ_ERR_NULL;
    }
    if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(out, 16) || !aligned(row_expert, 4)) {
        report(fn, MMQ_ERR_ALIGN, "xq, wq and out must be 16-byte aligned, row_expert 4-byte aligned");
        return MMQ_ERR_ALIGN;
    }
    if (!tc_available()) {
        report(fn, MMQ_ERR_LAUNCH, "the grouped contraction needs the tcgen05 tensor cores");
        return MMQ_ERR_LAUNCH;
    }
    const bool use_tc = current_path() == MMQ_PATH_TC;
    if (use_tc && fmt == FMT_Q6_K) {
        report(fn, MMQ_ERR_ARG, "the converter tensor-core kernel takes Q8_0, Q4_K and Q5_K (Q6_K: the expanded path)");
        return MMQ_ERR_ARG;
    }
    int taken = MMQ_PATH_EXPAND;
    st = grouped_launch_path(fmt, xq, row_expert, R, wq, E, N, K, out, static_cast<cudaStream_t>(stream),
                             current_path(), &taken);
    if (st == MMQ_OK) t_last_path = taken;
    return st;
}

}  // namespace
}  // namespace mmq

using namespace mmq;

extern "C" {

const char* mmq_status_string(int status) {
    switch (status) {
        case MMQ_OK: return "MMQ_OK";
        case MMQ_ERR_SHAPE: return "MMQ_ERR_SHAPE";
        case MMQ_ERR_K_MULTIPLE: return "MMQ_ERR_K_MULTIPLE";
        case MMQ_ERR_NULL: return "MMQ_ERR_NULL";
        case MMQ_ERR_ALIGN: return "MMQ_ERR_ALIGN";
        case MMQ_ERR_SMEM: return "MMQ_ERR_SMEM";
        case MMQ_ERR_LAUNCH: return "MMQ_ERR_LAUNCH";
        case MMQ_ERR_TIMEOUT: return "MMQ_ERR_TIMEOUT";
        case MMQ_ERR_CUDA: return "MMQ_ERR_CUDA";
        case MMQ_ERR_ARG: return "MMQ_ERR_ARG";
        case MMQ_ERR_NOMEM: return "MMQ_ERR_NOMEM";
        default: return "MMQ_ERR_UNKNOWN";
    }
}

size_t mmq_q8_1_bytes(int64_t M, int64_t K) {
    if (M < 0 || K < 0 || K % QK != 0) return 0;
    return (size_t)M * (size_t)(K / QK) * Q8_1_BYTES;
}

size_t mmq_weight_row_bytes(int fmt, int64_t K) {
    if (K < 0) return 0;
    if (fmt == FMT_Q8_0 && K % QK == 0) return (size_t)(K / QK) * Q8_0_BYTES;
    if (fmt == FMT_Q4_K && K % QK_K == 0) return (size_t)(K / QK_K) * Q4_K_BYTES;
    if (fmt == FMT_Q5_K && K % QK_K == 0) return (size_t)(K / QK_K) * Q5_K_BYTES;
    if (fmt == FMT_Q6_K && K % QK_K == 0) return (size_t)(K / QK_K) * Q6_K_BYTES;
    return 0;
}

int mmq_quantize_q8_1(const float* x, int64_t M, int64_t K, void* xq, void* stream) {
    const char* fn = "mmq_quantize_q8_1";
    int st = check_mk(fn, M, 1, K, QK);
    if (st) return st;
    if (!x || !xq) {
        report(fn, MMQ_ERR_NULL, "x and xq must be non-NULL");
        return MMQ_ERR_NULL;
    }
    if (!aligned(x, 16) || !aligned(xq, 4)) {
        report(fn, MMQ_ERR_ALIGN, "x must be 16-byte and xq 4-byte aligned");
        return MMQ_ERR_ALIGN;
    }
    return quantize_launch(x, M, K, xq, static_cast<cudaStream_t>(stream));
}

int mmq_gemm_q8_0(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, void* stream) {
    return contraction("mmq_gemm_q8_0", FMT_Q8_0, xq, wq, M, N, K, out, nullptr, stream);
}

int mmq_gemm_q4_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, void* stream) {
    return contraction("mmq_gemm_q4_k", FMT_Q4_K, xq, wq, M, N, K, out, nullptr, stream);
}

int mmq_gemm_q5_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, void* stream) {
    return contraction("mmq_gemm_q5_k", FMT_Q5_K, xq, wq, M, N, K, out, nullptr, stream);
}

int mmq_linear_q5_k(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream) {
    return linear("mmq_linear_q5_k", FMT_Q5_K, x, M, K, wq, N, xq, out, stream);
}

int mmq_debug_block_dots_q5_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, int32_t* dots,
                              void* stream) {
    return contraction("mmq_debug_block_dots_q5_k", FMT_Q5_K, xq, wq, M, N, K, nullptr, dots, stream);
}

int mmq_gemm_q6_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out, void* stream) {
    return contraction("mmq_gemm_q6_k", FMT_Q6_K, xq, wq, M, N, K, out, nullptr, stream);
}

int mmq_linear_q6_k(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream) {
    return linear("mmq_linear_q6_k", FMT_Q6_K, x, M, K, wq, N, xq, out, stream);
}

int mmq_debug_block_dots_q6_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, int32_t* dots,
                              void* stream) {
    return contraction("mmq_debug_block_dots_q6_k", FMT_Q6_K, xq, wq, M, N, K, nullptr, dots, stream);
}

int mmq_linear_q8_0(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream) {
    return linear("mmq_linear_q8_0", FMT_Q8_0, x, M, K, wq, N, xq, out, stream);
}

int mmq_linear_q4_k(const float* x, int64_t M, int64_t K, const void* wq, int64_t N, void* xq, float* out,
                    void* stream) {
    return linear("mmq_linear_q4_k", FMT_Q4_K, x, M, K, wq, N, xq, out, stream);
}

int mmq_gemm_grouped_q8_0(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream) {
    return grouped("mmq_gemm_grouped_q8_0", FMT_Q8_0, xq, row_expert, R, wq, E, N, K, out, stream);
}

int mmq_gemm_grouped_q4_k(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream) {
    return grouped("mmq_gemm_grouped_q4_k", FMT_Q4_K, xq, row_expert, R, wq, E, N, K, out, stream);
}

int mmq_gemm_grouped_q6_k(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream) {
    return grouped("mmq_gemm_grouped_q6_k", FMT_Q6_K, xq, row_expert, R, wq, E, N, K, out, stream);
}

int mmq_gemm_grouped_q5_k(const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                          int64_t K, float* out, void* stream) {
    return grouped("mmq_gemm_grouped_q5_k", FMT_Q5_K, xq, row_expert, R, wq, E, N, K, out, stream);
}

int mmq_debug_block_dots_q8_0(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, int32_t* dots,
                              void* stream) {
    return contraction("mmq_debug_block_dots_q8_0", FMT_Q8_0, xq, wq, M, N, K, nullptr, dots, stream);
}

int mmq_debug_block_dots_q4_k(const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, int32_t* dots,
                              void* stream) {
    return contraction("mmq_debug_block_dots_q4_k", FMT_Q4_K, xq, wq, M, N, K, nullptr, dots, stream);
}

int mmq_gemm_noalloc(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                     void* stream) {
    const char* fn = "mmq_gemm_noalloc";
    if (fmt != FMT_Q8_0 && fmt != FMT_Q4_K && fmt != FMT_Q5_K && fmt != FMT_Q6_K) {
        report(fn, MMQ_ERR_ARG, "fmt must be 0 (Q8_0), 1 (Q4_K), 2 (Q5_K) or 3 (Q6_K)");
        return MMQ_ERR_ARG;
    }
    int st = check_mk(fn, M, N, K, is_superblock(fmt) ? QK_K : QK);
    if (st) return st;
    if (!xq || !wq || !out) {
        report(fn, MMQ_ERR_NULL, "xq, wq and out must be non-NULL");
        return MMQ_ERR_NULL;
    }
    if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(out, 16)) {
        report(fn, MMQ_ERR_ALIGN, "xq, wq and out must be 16-byte aligned");
        return MMQ_ERR_ALIGN;
    }
    st = tcx_launch_noalloc(fmt, xq, wq, M, N, K, out, static_cast<cudaStream_t>(stream));
    if (st == MMQ_OK) t_last_path = MMQ_PATH_EXPAND;
    return st;
}

int mmq_debug_product_dots(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, int32_t* dots,
                           void* stream) {
    const char* fn = "mmq_debug_product_dots";
    if (fmt != FMT_Q8_0 && fmt != FMT_Q4_K && fmt != FMT_Q5_K && fmt != FMT_Q6_K) {
        report(fn, MMQ_ERR_ARG, "fmt must be 0 (Q8_0), 1 (Q4_K), 2 (Q5_K) or 3 (Q6_K)");
        return MMQ_ERR_ARG;
    }
    int st = check_mk(fn, M, N, K, QK_K);
    if (st) return st;
    if (!xq || !wq || !dots) {
        report(fn, MMQ_ERR_NULL, "xq, wq and dots must be non-NULL");
        return MMQ_ERR_NULL;
    }
    if (!aligned(xq, 16) || !aligned(wq, 16) || !aligned(dots, 16)) {
        report(fn, MMQ_ERR_ALIGN, "xq, wq and dots must be 16-byte aligned");
        return MMQ_ERR_ALIGN;
    }
    st = tcx_launch(fmt, xq, wq, M, N, K, nullptr, dots, static_cast<cudaStream_t>(stream), true);
    if (st == MMQ_OK) t_last_path = MMQ_PATH_EXPAND;
    return st;
}

int mmq_debug_refuse_smem(int on) { return g_refuse_smem.exchange(on ? 1 : 0); }

int mmq_debug_small_route(int route) {
    if (route < SMALL_ROUTE_AUTO || route > SMALL_ROUTE_MMA) return MMQ_ERR_ARG;
    return small_set_route(route);
}

int mmq_debug_small_grid(int fmt, int64_t M, int64_t N, int64_t K, int32_t* boxes, int32_t* splits) {
    const char* fn = "mmq_debug_small_grid";
    if (fmt != FMT_Q8_0 && fmt != FMT_Q4_K && fmt != FMT_Q5_K) {
        report(fn, MMQ_ERR_ARG, "fmt must be 0 (Q8_0), 1 (Q4_K) or 2 (Q5_K)");
        return MMQ_ERR_ARG;
    }
    const int st = check_mk(fn, M, N, K, QK_K);
    if (st) return st;
    if (!boxes || !splits) {
        report(fn, MMQ_ERR_NULL, "boxes and splits must be non-NULL");
        return MMQ_ERR_NULL;
    }
    small_stream_grid(fmt, M, N, K, boxes, splits);
    return MMQ_OK;
}

int mmq_debug_small_ksplit(int splits, int boxes) {
    if (splits < 0 || splits > 8 || boxes < 0 || boxes > 4) return MMQ_ERR_ARG;
    small_set_ksplit(splits, boxes);
    return MMQ_OK;
}

int mmq_debug_expand_tiling(int fmt, int64_t M, int64_t N, int64_t K, int32_t* tile_n, int32_t* splits) {
    const char* fn = "mmq_debug_expand_tiling";
    if (fmt != FMT_Q8_0 && fmt != FMT_Q4_K && fmt != FMT_Q5_K && fmt != FMT_Q6_K) {
        report(fn, MMQ_ERR_ARG, "fmt must be 0 (Q8_0), 1 (Q4_K), 2 (Q5_K) or 3 (Q6_K)");
        return MMQ_ERR_ARG;
    }
    const int st = check_mk(fn, M, N, K, QK_K);
    if (st) return st;
    if (!tile_n || !splits) {
        report(fn, MMQ_ERR_NULL, "tile_n and splits must be non-NULL");
        return MMQ_ERR_NULL;
    }
    *tile_n = tcx_tile_n(fmt, M, N);
    *splits = tcx_splits(fmt, M, N, K);
    return MMQ_OK;
}

int mmq_debug_set_wait_limit(int64_t ns) {
    return tcx_set_wait_limit(ns >= 0 ? (unsigned long long)ns : 2000000000ull);
}

int mmq_set_path(int path) {
    if (path != MMQ_PATH_AUTO && path != MMQ_PATH_SMALL && path != MMQ_PATH_TC && path != MMQ_PATH_EXPAND)
        return MMQ_ERR_ARG;
    const int prev = current_path();
    g_path.store(path);
    return prev;
}

int mmq_last_path(void) { return t_last_path; }

int mmq_get_device_error(void* stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        fprintf(stderr, "libmmq: mmq_get_device_error: %s\n", cudaGetErrorString(e));
        return MMQ_ERR_CUDA;
    }
    const unsigned bits = tc_take_error() | tcx_take_error() | small_take_error();
    return (bits & ERR_TIMEOUT) ? MMQ_ERR_TIMEOUT : MMQ_OK;
}

}  // extern "C"
