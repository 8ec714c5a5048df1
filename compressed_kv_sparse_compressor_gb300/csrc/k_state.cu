// State initialisation (K3), raw-ring commit (K7) and logical-order
// checkpoint gather (K8).  All three are plain HBM copies / fills: coalesced
// 16-byte accesses, grid-stride loops over a grid of a few waves of the SMs.
#include <cuda_bf16.h>

#include "ds4c_internal.cuh"

namespace ds4c {
namespace {

__global__ void fill_kernel(float *__restrict__ p, size_t n, float v) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    if (((uintptr_t)p & 15) == 0) {
        float4 v4 = make_float4(v, v, v, v);
        size_t n4 = n / 4;
        for (size_t j = i; j < n4; j += stride) reinterpret_cast<float4 *>(p)[j] = v4;
        for (size_t j = n4 * 4 + i; j < n; j += stride) p[j] = v;
    } else {
        for (size_t j = i; j < n; j += stride) p[j] = v;
    }
}

// Ring commit, "Metal グラフと圧縮 KV の実装を読む" §2: raw_kv keeps the most
// recent swa rows; slot p % swa holds position p.  Prefill (n_seq == 1): the
// last min(n_tok, S) rows of the chunk.  Decode: one row per sequence.
__global__ void ring_commit_kernel(float *__restrict__ ring, const float *__restrict__ raw_new, int D, int S,
                                   int n_seq, int n_tok, uint64_t pos0, DecodePos dp) {
    pdl_wait();
    pdl_launch_dependents();
    const int r = blockIdx.x;                  // row within the committed set
    uint64_t p;
    const float *src;
    float *dst;
    if (n_seq == 1) {
        uint64_t end = pos0 + (uint64_t)n_tok;
        uint64_t start = (end - pos0 > (uint64_t)S) ? end - (uint64_t)S : pos0;
        p = start + (uint64_t)r;
        if (p >= end) return;
        src = raw_new + (size_t)(p - pos0) * D;
        dst = ring + (size_t)(p % (uint64_t)S) * D;
    } else {
        if (r >= n_seq) return;
        p = dp.pos[r];
        src = raw_new + (size_t)r * D;
        dst = ring + ((size_t)r * S + (size_t)(p % (uint64_t)S)) * D;
    }
    for (int j = threadIdx.x * 4; j < D; j += blockDim.x * 4)
        *reinterpret_cast<float4 *>(dst + j) = *reinterpret_cast<const float4 *>(src + j);
}

// Checkpoint gather, "【#4】ds4.c を読み解く" §5-§7.  Segment 0 (the raw ring)
// maps destination row i to slot (pos - n_live + i) % S; the other segments
// are contiguous copies.  blockIdx.y picks the segment.
__global__ void gather_kernel(GatherArgs a, int vec) {
    const int s = blockIdx.y;
    if (s > a.n_seg) return;
    size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    if (s == 0) {
        size_t n = (size_t)a.n_live * a.D;
        uint64_t first = a.pos - (uint64_t)a.n_live;
        for (size_t i = tid * (vec ? 4 : 1); i < n; i += stride * (vec ? 4 : 1)) {
            size_t row = i / a.D, col = i % a.D;
            size_t slot = (size_t)((first + row) % (uint64_t)a.S);
            const float *src = a.ring + slot * a.D + col;
            if (vec) *reinterpret_cast<float4 *>(a.dst + i) = *reinterpret_cast<const float4 *>(src);
            else a.dst[i] = *src;
        }
        return;
    }
    const GatherSeg g = a.seg[s - 1];
    float *dst = a.dst + g.dst_off;
    if (vec) {
        size_t n4 = (size_t)g.n / 4;
        for (size_t i = tid; i < n4; i += stride)
            reinterpret_cast<float4 *>(dst)[i] = reinterpret_cast<const float4 *>(g.src)[i];
        for (size_t i = n4 * 4 + tid; i < (size_t)g.n; i += stride) dst[i] = g.src[i];
    } else {
        for (size_t i = tid; i < (size_t)g.n; i += stride) dst[i] = g.src[i];
    }
}

// Restore of a checkpoint (the inverse of gather_kernel): destination row i of
// the raw segment goes to slot (pos - n_live + i) % S; the other segments are
// contiguous copies.  blockIdx.y picks the segment.
__global__ void scatter_kernel(ScatterArgs a, int vec) {
    const int s = blockIdx.y;
    if (s > a.n_seg) return;
    size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t stride = (size_t)gridDim.x * blockDim.x;
    if (s == 0) {
        size_t n = (size_t)a.n_live * a.D;
        uint64_t first = a.pos - (uint64_t)a.n_live;
        for (size_t i = tid * (vec ? 4 : 1); i < n; i += stride * (vec ? 4 : 1)) {
            size_t row = i / a.D, col = i % a.D;
            size_t slot = (size_t)((first + row) % (uint64_t)a.S);
            float *dst = a.ring + slot * a.D + col;
            if (vec) *reinterpret_cast<float4 *>(dst) = *reinterpret_cast<const float4 *>(a.src + i);
            else *dst = a.src[i];
        }
        return;
    }
    const ScatterSeg g = a.seg[s - 1];
    const float *src = a.src + g.src_off;
    if (vec) {
        size_t n4 = (size_t)g.n / 4;
        for (size_t i = tid; i < n4; i += stride)
            reinterpret_cast<float4 *>(g.dst)[i] = reinterpret_cast<const float4 *>(src)[i];
        for (size_t i = n4 * 4 + tid; i < (size_t)g.n; i += stride) g.dst[i] = src[i];
    } else {
        for (size_t i = tid; i < (size_t)g.n; i += stride) g.dst[i] = src[i];
    }
}

// hi = bf16(x), lo = bf16(x - hi) of each element, into [row][2][D]
__global__ void split_rows_kernel(uint16_t *__restrict__ split, const float *__restrict__ rows, int64_t n, int D) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / D, c = i % D;
        const float x = rows[i];
        const __nv_bfloat16 h = __float2bfloat16_rn(x);
        const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
        split[(r * 2) * D + c] = *reinterpret_cast<const uint16_t *>(&h);
        split[(r * 2 + 1) * D + c] = *reinterpret_cast<const uint16_t *>(&l);
    }
}

int sm_count() {
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

}  // namespace

cudaError_t launch_fill(float *p, size_t n, float v, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    size_t blocks = (n / 4 + 255) / 256;
    size_t cap = (size_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    fill_kernel<<<(unsigned)blocks, 256, 0, s>>>(p, n, v);
    return cudaGetLastError();
}

cudaError_t launch_ring_commit(float *ring, const float *raw_new, int D, int S, int n_seq, int n_tok,
                               uint64_t pos0, const DecodePos *p, cudaStream_t s) {
    int rows = (n_seq == 1) ? (n_tok < S ? n_tok : S) : n_seq;
    if (rows <= 0) return cudaSuccess;
    int threads = D / 4 < 128 ? D / 4 : 128;
    DecodePos dp{};
    if (n_seq > 1) dp = *p;
    return launch_pdl(ring_commit_kernel, dim3(rows), dim3(threads), 0, s, ring, raw_new, D, S, n_seq, n_tok, pos0, dp);
}

cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s) {
    bool vec = ((uintptr_t)a.dst & 15) == 0 && ((uintptr_t)a.ring & 15) == 0 && (a.D % 4) == 0;
    for (int i = 0; i < a.n_seg; i++)
        vec = vec && ((uintptr_t)a.seg[i].src & 15) == 0 && (a.seg[i].dst_off % 4) == 0;
    int64_t biggest = a.n_live * a.D;
    for (int i = 0; i < a.n_seg; i++) biggest = a.seg[i].n > biggest ? a.seg[i].n : biggest;
    int64_t blocks = (biggest / 4 + 255) / 256;
    int64_t cap = (int64_t)sm_count() * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    dim3 grid((unsigned)blocks, (unsigned)(a.n_seg + 1));
    gather_kernel<<<grid, 256, 0, s>>>(a, vec ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_scatter(const ScatterArgs &a, cudaStream_t s) {
    bool vec = ((uintptr_t)a.src & 15) == 0 && ((uintptr_t)a.ring & 15) == 0 && (a.D % 4) == 0;
    for (int i = 0; i < a.n_seg; i++)
        vec = vec && ((uintptr_t)a.seg[i].dst & 15) == 0 && (a.seg[i].src_off % 4) == 0;
    int64_t biggest = a.n_live * a.D;
    for (int i = 0; i < a.n_seg; i++) biggest = a.seg[i].n > biggest ? a.seg[i].n : biggest;
    int64_t blocks = (biggest / 4 + 255) / 256;
    int64_t cap = (int64_t)sm_count() * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    dim3 grid((unsigned)blocks, (unsigned)(a.n_seg + 1));
    scatter_kernel<<<grid, 256, 0, s>>>(a, vec ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_split_rows(uint16_t *split, const float *rows, int64_t n_rows, int D, cudaStream_t s) {
    const int64_t n = n_rows * D;
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    split_rows_kernel<<<(unsigned)blocks, 256, 0, s>>>(split, rows, n, D);
    return cudaGetLastError();
}

}  // namespace ds4c
