// FP32 FMA rate of this GPU, the denominator of the indexer score's roofline
// (the score is an in-order fp32 fmaf chain per output, on the CUDA cores).
// Every thread runs independent fmaf chains in registers and stores one sum,
// so the kernel does no memory traffic worth counting.
#include "ds4c_internal.cuh"

namespace ds4c {
namespace {

constexpr int PROBE_THREADS = 256;
constexpr int PROBE_CHAINS = 16;

__global__ void __launch_bounds__(PROBE_THREADS) fma_probe_kernel(float *__restrict__ out, int iters, float b) {
    float acc[PROBE_CHAINS];
#pragma unroll
    for (int i = 0; i < PROBE_CHAINS; i++) acc[i] = threadIdx.x * 1e-3f + (float)i;
    float x = 1.0f + threadIdx.x * 1e-6f;
    for (int it = 0; it < iters; it++) {
#pragma unroll
        for (int i = 0; i < PROBE_CHAINS; i++) acc[i] = __fmaf_rn(x, b, acc[i]);
        x = __fmaf_rn(x, 1.0000001f, 1e-7f);
    }
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < PROBE_CHAINS; i++) sum += acc[i];
    out[(size_t)blockIdx.x * PROBE_THREADS + threadIdx.x] = sum;
}

}  // namespace

double fma_probe_flops(uint32_t blocks, uint32_t iters) {
    return 2.0 * (double)blocks * PROBE_THREADS * (double)iters * (PROBE_CHAINS + 1);
}

cudaError_t launch_fma_probe(uint32_t blocks, uint32_t iters, float *out, cudaStream_t s) {
    fma_probe_kernel<<<blocks, PROBE_THREADS, 0, s>>>(out, (int)iters, 0.999999f);
    return cudaGetLastError();
}

}  // namespace ds4c
