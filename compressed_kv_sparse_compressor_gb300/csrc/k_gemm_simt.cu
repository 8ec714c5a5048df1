// Projection GEMM on the CUDA cores (K1s): C[m][n] = sum_k A[m][k] * B[n][k]
// with fp32 accumulation.  Used for fp32 weights ("one ratio-4 layer, fp32
// throughout") and for shapes the tcgen05 kernel does not take.  Up to four
// weight matrices (wkv, wgate of both lanes) share one launch: blockIdx.z picks
// the group.  64x64 output tile per 256-thread block, 4x4 per thread, 32-deep
// k slices staged in shared memory.
#include <cuda_bf16.h>

#include "ds4c_internal.cuh"

namespace ds4c {
namespace {

constexpr int BM = 64, BN = 64, BK = 32;

template <int DT>
__device__ __forceinline__ float load_elem(const void *p, size_t i) {
    if (DT == DS4C_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    return reinterpret_cast<const float *>(p)[i];
}

template <int DT>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs a) {
    const GemmGroup g = a.g[blockIdx.z];
    const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
    if (n0 >= g.N) return;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < a.K; k0 += BK) {
        for (int e = threadIdx.x; e < BM * BK; e += 256) {
            int r = e / BK, kk = e % BK;
            int m = m0 + r, k = k0 + kk;
            As[kk][r] = (m < a.M && k < a.K) ? load_elem<DT>(a.A, (size_t)m * a.K + k) : 0.f;
            int n = n0 + r;
            Bs[kk][r] = (n < g.N && k < a.K) ? load_elem<DT>(g.B, (size_t)n * a.K + k) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < BK; kk++) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; i++) av[i] = As[kk][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; j++) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        int m = m0 + ty * 4 + i;
        if (m >= a.M) continue;
#pragma unroll
        for (int j = 0; j < 4; j++) {
            int n = n0 + tx * 4 + j;
            if (n < g.N) g.C[(size_t)m * g.ldc + n] = acc[i][j];
        }
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const GemmArgs &a, cudaStream_t s) {
    int maxN = 0;
    for (int i = 0; i < a.n_groups; i++) maxN = a.g[i].N > maxN ? a.g[i].N : maxN;
    dim3 grid((maxN + BN - 1) / BN, (a.M + BM - 1) / BM, a.n_groups);
    if (a.dtype == DS4C_BF16) gemm_simt_kernel<DS4C_BF16><<<grid, 256, 0, s>>>(a);
    else gemm_simt_kernel<DS4C_F32><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace ds4c
