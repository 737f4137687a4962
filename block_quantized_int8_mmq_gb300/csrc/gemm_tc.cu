// tcgen05 tensor-core MMQ (placeholder until the kernel lands).
#include "common.cuh"

namespace mmq {

bool tc_available() { return false; }

int tc_launch(int, const void*, const void*, int64_t, int64_t, int64_t, float*, int32_t*, cudaStream_t) {
    report("mmq_gemm (tc)", MMQ_ERR_ARG, "tensor-core path not built");
    return MMQ_ERR_ARG;
}

unsigned tc_take_error() { return 0; }

}  // namespace mmq
