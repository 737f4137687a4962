// f32 -> q8_1 activation quantization ("13 . r7-r8 raw-byte MMQ kernel", sec. 3.2, the
// quantize pass: tree-reduced block amax, scale, round, clamp, block sum).
//
// HBM-bound: 4 bytes read and 1.125 bytes written per value.  The input is treated as
// one flat array of M*K/32 blocks (rows are contiguous), so a warp streams 1 KiB of
// contiguous input per step.  Four lanes own one 32-value block, eight values each
// (two 16-byte loads); amax and the code sum are reduced across the four lanes with
// shuffles.  amax is exact under any association, so the tree order changes nothing.
//
// The arithmetic of one block (bit-exact: IEEE divisions, ties to even, s = f16(d * S)) is
// quantize_q8_1_part, shared with the fused quantize-and-expand kernel.
#include <stdio.h>

#include "common.cuh"
#include "ptx.cuh"
#include "quant_block.cuh"

namespace mmq {
namespace {

constexpr int QUANT_THREADS = 256;
constexpr int BLOCKS_PER_WARP = 8;  // 32 lanes / 4 lanes per block

__global__ void __launch_bounds__(QUANT_THREADS)
k_quantize_q8_1(const float* __restrict__ x, uint8_t* __restrict__ y, long long nblk) {
    const int lane = threadIdx.x & 31;
    const int sub = lane >> 2;   // block within the warp's group of 8
    const int part = lane & 3;   // which 8 values of the block
    const long long warp = ((long long)blockIdx.x * QUANT_THREADS + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * QUANT_THREADS) >> 5;
    // programmatic dependent: x may be the previous kernel's output
    ptx::grid_dep_wait();
    ptx::grid_dep_launch_dependents();

    for (long long base = warp * BLOCKS_PER_WARP; base < nblk; base += nwarps * BLOCKS_PER_WARP) {
        const long long g = base + sub;
        const bool valid = g < nblk;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (valid) {
            const float4* src = reinterpret_cast<const float4*>(x + g * QK + part * 8);
            a = __ldcs(src);
            b = __ldcs(src + 1);
        }
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t w0, w1, hdr;
        quantize_q8_1_part(v, w0, w1, hdr);
        if (valid) {
            uint8_t* dst = y + g * Q8_1_BYTES;
            if (part == 0) *reinterpret_cast<uint32_t*>(dst) = hdr;
            uint32_t* q32 = reinterpret_cast<uint32_t*>(dst + 4 + part * 8);
            q32[0] = w0;
            q32[1] = w1;
        }
    }
}

}  // namespace

int quantize_launch(const float* x, int64_t M, int64_t K, void* xq, cudaStream_t s) {
    const long long nblk = (long long)M * (K / QK);
    const long long per_cta = (QUANT_THREADS / 32) * BLOCKS_PER_WARP;
    long long grid = (nblk + per_cta - 1) / per_cta;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = (long long)(sms > 0 ? sms : 152) * 16;
    if (grid > cap) grid = cap;
    {
        ProfScope ps("k_quantize_q8_1", s);
        return pdl_status(launch_pdl(k_quantize_q8_1, dim3((unsigned)grid), dim3(QUANT_THREADS), 0, s, x,
                                     static_cast<uint8_t*>(xq), nblk),
                          "mmq_quantize_q8_1");
    }
}

}  // namespace mmq
