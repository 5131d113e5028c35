// Scaled FP8 GEMM (placeholder until the tcgen05 kernels land).
#include "fp8q_internal.cuh"

namespace fp8q {

__device__ unsigned int g_device_errors = 0;

fp8q_status read_device_errors(unsigned int* flags, cudaStream_t s) {
    if (cudaStreamSynchronize(s) != cudaSuccess) return FP8Q_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_errors, sizeof(v)) != cudaSuccess) return FP8Q_ERR_CUDA;
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_errors, &zero, sizeof(zero)) != cudaSuccess) return FP8Q_ERR_CUDA;
    *flags = v;
    return FP8Q_OK;
}

fp8q_status launch_gemm(const GemmOperand&, const GemmOperand&, void*, int, int64_t, int64_t, int64_t,
                        cudaStream_t) {
    return FP8Q_ERR_UNSUPPORTED;
}

}  // namespace fp8q
