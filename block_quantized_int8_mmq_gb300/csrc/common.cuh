// Shared device/host helpers of libmmq (sm_103a).  Block-format constants follow the
// q8_1 / Q8_0 / Q4_K layouts described in include/mmq.h.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mmq.h"

namespace mmq {

constexpr int QK = 32;           // values per q8_1 / Q8_0 block and per Q4_K sub-block
constexpr int QK_K = 256;        // values per Q4_K super-block
constexpr int Q8_1_BYTES = 36;   // f16 d, f16 s, int8 q[32]
constexpr int Q8_0_BYTES = 34;   // f16 d, int8 q[32]
constexpr int Q4_K_BYTES = 144;  // f16 d, f16 dmin, 12 scale bytes, 128 nibble bytes
constexpr int Q5_K_BYTES = 176;  // f16 d, f16 dmin, 12 scale bytes, 32 high-bit bytes, 128 nibble bytes
constexpr int Q6_K_BYTES = 210;  // 128 low-nibble bytes, 64 bytes of 2-bit high parts, 16 int8 scales, f16 d

enum WeightFormat { FMT_Q8_0 = 0, FMT_Q4_K = 1, FMT_Q5_K = 2, FMT_Q6_K = 3 };
// K-quant super-block formats with mins (256 values, eight 32-value sub-blocks with 6-bit
// scales and mins, a min term per sub-block): Q4_K and Q5_K
__host__ __device__ constexpr bool is_kquant(int fmt) { return fmt == FMT_Q4_K || fmt == FMT_Q5_K; }
// every format stored in 256-value super-blocks (K % 256 == 0): the K-quants with mins and
// Q6_K (sixteen 16-value groups with int8 scales, values centred on 32, no min term)
__host__ __device__ constexpr bool is_superblock(int fmt) { return is_kquant(fmt) || fmt == FMT_Q6_K; }
__host__ __device__ constexpr int kq_bytes(int fmt) {
    return fmt == FMT_Q6_K ? Q6_K_BYTES : fmt == FMT_Q5_K ? Q5_K_BYTES : Q4_K_BYTES;
}
// byte offset of the 128 nibble bytes in a super-block (Q5_K: after the 32 high-bit bytes)
__host__ __device__ constexpr int kq_qs_off(int fmt) { return fmt == FMT_Q5_K ? 48 : 16; }

// Error bits a kernel may set in its translation unit's device error word.
constexpr unsigned ERR_TIMEOUT = 1u;

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half((unsigned short)(bits16 & 0xffffu)));
}

// Q4_K: 6-bit sub-scale and sub-min of sub-block j (0..7) from the 12 packed scale
// bytes, given as three little-endian words s0 = bytes 0..3, s1 = 4..7, s2 = 8..11.
// Sub-blocks 0..3: low 6 bits of byte j (scale) and byte j+4 (min).  Sub-blocks 4..7:
// low nibble / high nibble of byte j+4 (scale / min low bits) and the top two bits of
// byte j-4 (scale) and byte j (min).
__device__ __forceinline__ void q4_k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j,
                                               int& sc, int& mn) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63;
        mn = (s1 >> (8 * j)) & 63;
    } else {
        const int i = j - 4;
        const uint32_t lo = (s2 >> (8 * i)) & 0xff;
        sc = (lo & 15) | (((s0 >> (8 * i + 6)) & 3) << 4);
        mn = (lo >> 4) | (((s1 >> (8 * i + 6)) & 3) << 4);
    }
}

}  // namespace mmq

// Host-side per-translation-unit hooks (defined in each .cu that owns kernels).
namespace mmq {
int quantize_launch(const float* x, int64_t M, int64_t K, void* xq, cudaStream_t s);
// which small-M kernel takes a shape with K % 256 == 0: the measured choice, the dp4a
// weight stream (up to four rows per pass) or the tensor-core stream (eight rows per pass;
// for Q6_K where K % 512 == 0 and N % 8 == 0).  small_set_route returns the previous setting.
enum SmallRoute { SMALL_ROUTE_AUTO = 0, SMALL_ROUTE_DP4A = 1, SMALL_ROUTE_MMA = 2 };
int small_set_route(int route);
int small_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                 int32_t* dots, cudaStream_t s);
int tc_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
              int32_t* dots, cudaStream_t s);
int tcx_launch(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
               int32_t* dots, cudaStream_t s, bool fold);
int tcx_linear_launch(int fmt, const float* x, void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                      cudaStream_t s);
int tcx_launch_noalloc(int fmt, const void* xq, const void* wq, int64_t M, int64_t N, int64_t K, float* out,
                       cudaStream_t s);
// K splits and tile width (weight rows) the expanded path's contraction takes for M x N x K
int tcx_splits(int fmt, int64_t M, int64_t N, int64_t K);
int tcx_tile_n(int fmt, int64_t M, int64_t N);
// bound of the expanded-path contraction's pipeline waits (device value; teardown drains
// keep their own fixed bound)
int tcx_set_wait_limit(unsigned long long ns);

constexpr int MAX_DEVICES = 64;  // per-device host caches are indexed by the device ordinal
// SM count, shared memory per SM and L2 bytes of the current device (queried once per
// device; GB300 values if the query fails)
struct DeviceShape {
    int sms = 0, smem_per_sm = 0, l2_bytes = 0;
};
DeviceShape device_shape();
// A kernel's dynamic shared-memory limit, raised once per device: cudaFuncSetAttribute
// applies to the device current when it is called.  ensure_smem returns MMQ_OK,
// MMQ_ERR_SMEM (refused, or refused on purpose by the test switch) or MMQ_ERR_CUDA.
struct SmemAttr {
    std::atomic<int> bytes[MAX_DEVICES];
};
int ensure_smem(const void* func, int bytes, SmemAttr& a);
int tc_grouped_launch(int fmt, const void* xs, const void* wq, int64_t R, int64_t E, int64_t N, int64_t K,
                      const int2* tiles, const int* ntiles, int64_t max_tiles, const int* row_end, const int* row_map,
                      float* out, cudaStream_t s);
// the expanded path's grouped contraction over the grouping (activation rows read from xq
// through perm; offsets[e + 1] = expert e's end in the sorted order)
int tcx_grouped_launch(int fmt, const void* xq, int64_t R, const void* wq, int64_t E, int64_t N, int64_t K,
                       const int2* tiles, const int* ntiles, int64_t max_tiles, const int* offsets, const int* perm,
                       float* out, cudaStream_t s, const char* fn);
// expert-grouped call: the grouping kernels, then the converter kernel (use_tc) or the
// expanded path
int grouped_launch(int fmt, const void* xq, const int32_t* row_expert, int64_t R, const void* wq, int64_t E, int64_t N,
                   int64_t K, float* out, cudaStream_t s, bool use_tc);
int scratch_alloc(size_t bytes, cudaStream_t s, void** p, const char* fn);
void scratch_free(void* p, cudaStream_t s);
unsigned tc_take_error();
unsigned tcx_take_error();
unsigned small_take_error();
bool make_byte_map(CUtensorMap* map, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
                   uint32_t box_rows, int elem_bytes);
void report(const char* fn, int status, const char* detail);
int launch_status(const char* fn);

// Launch as a programmatic dependent of the previous kernel on the stream: the kernel may be
// scheduled while that kernel drains, if that kernel allows it (griddepcontrol.launch_dependents);
// the kernel itself must execute griddepcontrol.wait before it reads anything the previous
// kernel may have written and before any global write.  Returns the launch's CUDA error.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// launch_status for a launch_pdl result: the error reported (and cleared) or MMQ_OK
inline int pdl_status(cudaError_t e, const char* fn) {
    if (e != cudaSuccess) {
        cudaGetLastError();
        report(fn, MMQ_ERR_LAUNCH, cudaGetErrorString(e));
        return MMQ_ERR_LAUNCH;
    }
    return launch_status(fn);
}

// Per-kernel timing (profile.cu): a ProfScope around a launch brackets it with two
// events on `s` while profiling is enabled.
bool profiling();
int prof_begin(const char* name, cudaStream_t s);
void prof_end(int slot, cudaStream_t s);
struct ProfScope {
    int slot = -1;
    cudaStream_t s;
    ProfScope(const char* name, cudaStream_t st) : s(st) {
        if (profiling()) slot = prof_begin(name, st);
    }
    ~ProfScope() {
        if (slot >= 0) prof_end(slot, s);
    }
};
}  // namespace mmq
