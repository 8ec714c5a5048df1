// Indexer score (K4) and top-k selection (K5) of ratio-4 layers
// ("Metal グラフと圧縮 KV の実装を読む" §6 indexer, §7 the attention reads the
// top-k list in ascending order and stops at the first row not yet visible).
//
// Score: s[t][c] = fmaf chain over i = 0..d-1 of q[t][i] * row[c][i], in
// float and in order, so that the selection is bit-exact against any other
// implementation of the same chain.  That fixes the arithmetic to the CUDA
// cores (a tensor-core MMA sums in its own order); the kernel is a register-
// blocked SIMT "GEMM" whose per-element k loop stays sequential.
//
// Top-k: radix select on order-preserving 32-bit keys (one CTA per query,
// keys resident in shared memory), then an ordered compaction that emits the
// selected indices in ascending order, ties at the threshold broken toward
// the lower index.
#include "ds4c_internal.cuh"

namespace ds4c {
namespace {

// ---------------------------------------------------------------------------
// K4 prefill: n_tok queries of one sequence, 64x64 (query x row) tile per
// 256-thread block, 4x4 per thread, d consumed in 32-wide slices in order.
// ---------------------------------------------------------------------------
constexpr int SB = 64, SK = 32;

__global__ void __launch_bounds__(256) score_prefill_kernel(IndexerArgs a) {
    const int j0 = blockIdx.y * SB, c0 = blockIdx.x * SB;
    const int jlast = min(j0 + SB, a.n_tok) - 1;
    const uint64_t vis_max = (a.pos0 + (uint64_t)jlast + 1) / 4;
    if ((uint64_t)c0 >= vis_max) return;
    __shared__ float Qs[SK][SB + 4];
    __shared__ float Rs[SK][SB + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; i++)
#pragma unroll
        for (int k = 0; k < 4; k++) acc[i][k] = 0.f;
    for (int i0 = 0; i0 < a.d; i0 += SK) {
        for (int e = threadIdx.x; e < SB * SK; e += 256) {
            const int r = e / SK, ii = e % SK;
            const int j = j0 + r, c = c0 + r;
            Qs[ii][r] = (j < a.n_tok) ? a.q[(size_t)j * a.d + i0 + ii] : 0.f;
            Rs[ii][r] = ((uint64_t)c < vis_max) ? a.rows[(size_t)c * a.d + i0 + ii] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int ii = 0; ii < SK; ii++) {
            float qv[4], rv[4];
#pragma unroll
            for (int i = 0; i < 4; i++) qv[i] = Qs[ii][ty * 4 + i];
#pragma unroll
            for (int k = 0; k < 4; k++) rv[k] = Rs[ii][tx * 4 + k];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int k = 0; k < 4; k++) acc[i][k] = __fmaf_rn(qv[i], rv[k], acc[i][k]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int j = j0 + ty * 4 + i;
        if (j >= a.n_tok) continue;
        const uint64_t vis = (a.pos0 + (uint64_t)j + 1) / 4;
#pragma unroll
        for (int k = 0; k < 4; k++) {
            const int c = c0 + tx * 4 + k;
            if ((uint64_t)c < vis) a.scores[(size_t)j * a.lds + c] = acc[i][k];
        }
    }
}

// ---------------------------------------------------------------------------
// K4 decode: one query per sequence; a 128-thread block scores 128 rows of
// its sequence, one row per thread.  Rows are staged through shared memory
// with a padded stride so the in-order reads are conflict-free.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) score_decode_kernel(IndexerArgs a, DecodePos dp) {
    extern __shared__ float sm[];
    const int b = blockIdx.y;
    const uint64_t vis = (dp.pos[b] + 1) / 4;
    const int c0 = blockIdx.x * 128;
    if ((uint64_t)c0 >= vis) return;
    const int d = a.d, ld = d + 1;
    float *qs = sm;                 // [d]
    float *rs = sm + d;             // [128][d+1]
    const float *rows = a.rows + (size_t)b * a.seq_stride;
    for (int i = threadIdx.x; i < d; i += 128) qs[i] = a.q[(size_t)b * d + i];
    const uint64_t left = vis - (uint64_t)c0;
    const int nrows = left < 128 ? (int)left : 128;
    for (int e = threadIdx.x; e < 128 * d; e += 128) {
        const int r = e / d, i = e % d;
        rs[r * ld + i] = (r < nrows) ? rows[(size_t)(c0 + r) * d + i] : 0.f;
    }
    __syncthreads();
    if (threadIdx.x < nrows) {
        float s = 0.f;
        const float *row = rs + threadIdx.x * ld;
        for (int i = 0; i < d; i++) s = __fmaf_rn(qs[i], row[i], s);
        a.scores[(size_t)b * a.lds + c0 + threadIdx.x] = s;
    }
}

// ---------------------------------------------------------------------------
// K5 top-k.
// ---------------------------------------------------------------------------
constexpr int TK_THREADS = 512;

__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s + 0.0f);          // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of a 0/1 flag over TK_THREADS threads.
__device__ __forceinline__ int block_excl_scan(int flag, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < TK_THREADS / 32; w++) {
        const int v = warp_tot[w];
        if (w < warp) before += v;
        tot += v;
    }
    __syncthreads();
    total = tot;
    return before + in_warp;
}

__global__ void __launch_bounds__(TK_THREADS) topk_kernel(IndexerArgs a, DecodePos dp) {
    extern __shared__ uint32_t keys[];
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[TK_THREADS / 32];
    __shared__ uint32_t sh_prefix;
    __shared__ int sh_remaining;
    const int q = blockIdx.x;
    const uint64_t pos = (a.n_seq == 1) ? a.pos0 + (uint64_t)q : dp.pos[q];
    const int V = (int)((pos + 1) / 4);
    const int k = a.k;
    int32_t *out = a.topk + (size_t)q * k;
    if (V <= k) {
        for (int i = threadIdx.x; i < k; i += TK_THREADS) out[i] = (i < V) ? i : -1;
        return;
    }
    const float *s = a.scores + (size_t)q * a.lds;
    for (int c = threadIdx.x; c < V; c += TK_THREADS) keys[c] = order_key(s[c]);
    if (threadIdx.x == 0) { sh_prefix = 0; sh_remaining = k; }
    __syncthreads();
    // Radix select, 8 bits per pass from the top: find the key K* of the k-th
    // largest element; `remaining` = how many elements equal to K* to keep.
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += TK_THREADS) hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = sh_prefix;
        const uint32_t hmask = (shift == 24) ? 0u : (0xffffffffu << (shift + 8));
        for (int c = threadIdx.x; c < V; c += TK_THREADS) {
            const uint32_t key = keys[c];
            if ((key & hmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int rem = sh_remaining;
            int bin = 255;
            for (; bin > 0; bin--) {
                const int h = (int)hist[bin];
                if (h >= rem) break;
                rem -= h;
            }
            sh_prefix = prefix | ((uint32_t)bin << shift);
            sh_remaining = rem;
        }
        __syncthreads();
    }
    const uint32_t kstar = sh_prefix;
    const int remaining = sh_remaining;
    // Ordered compaction: keep key > K*, and the first `remaining` (by index)
    // of key == K*.
    int eq_run = 0, sel_run = 0;
    for (int base = 0; base < V; base += TK_THREADS) {
        const int c = base + threadIdx.x;
        const uint32_t key = (c < V) ? keys[c] : 0u;
        const int gt = (c < V) && key > kstar;
        const int eq = (c < V) && key == kstar;
        int eq_tot;
        const int eq_rank = eq_run + block_excl_scan(eq, warp_tot, eq_tot);
        const int sel = gt || (eq && eq_rank < remaining);
        int sel_tot;
        const int slot = sel_run + block_excl_scan(sel, warp_tot, sel_tot);
        if (sel) out[slot] = c;
        eq_run += eq_tot;
        sel_run += sel_tot;
    }
}

}  // namespace

cudaError_t launch_indexer_prefill(const IndexerArgs &a, cudaStream_t s) {
    const uint64_t vis_max = (a.pos0 + (uint64_t)a.n_tok) / 4;
    if (a.n_tok <= 0) return cudaSuccess;
    if (vis_max > 0) {
        dim3 grid((unsigned)((vis_max + SB - 1) / SB), (unsigned)((a.n_tok + SB - 1) / SB));
        score_prefill_kernel<<<grid, 256, 0, s>>>(a);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(uint32_t) * (size_t)(vis_max > 0 ? vis_max : 1);
    cudaError_t e = ensure_dyn_smem(topk_kernel, smem);
    if (e != cudaSuccess) return e;
    DecodePos dp{};
    topk_kernel<<<a.n_tok, TK_THREADS, smem, s>>>(a, dp);
    return cudaGetLastError();
}

cudaError_t launch_indexer_decode(const IndexerArgs &a, const DecodePos &p, cudaStream_t s) {
    uint64_t vis_max = 0;
    for (int b = 0; b < a.n_seq; b++) vis_max = ((p.pos[b] + 1) / 4 > vis_max) ? (p.pos[b] + 1) / 4 : vis_max;
    if (vis_max > 0) {
        dim3 grid((unsigned)((vis_max + 127) / 128), (unsigned)a.n_seq);
        const size_t smem = sizeof(float) * ((size_t)a.d + 128 * ((size_t)a.d + 1));
        cudaError_t e = ensure_dyn_smem(score_decode_kernel, smem);
        if (e != cudaSuccess) return e;
        score_decode_kernel<<<grid, 128, smem, s>>>(a, p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = sizeof(uint32_t) * (size_t)(vis_max > 0 ? vis_max : 1);
    cudaError_t e2 = ensure_dyn_smem(topk_kernel, smem);
    if (e2 != cudaSuccess) return e2;
    topk_kernel<<<a.n_seq, TK_THREADS, smem, s>>>(a, p);
    return cudaGetLastError();
}

}  // namespace ds4c
