// Sparse sliding-window attention (K6), "Metal グラフと圧縮 KV の実装を読む" §7
// (kernel_dsv4_indexed_mixed_attention_heads8): one online softmax per query
// and head over the raw window rows and the compressed rows the layer's ratio
// selects.  K = V = the stored row; all H heads share it (one KV head), so a
// CTA handles one query token for all heads and streams its rows once.
//
// This is the CUDA-core formulation: Q [H][D] and a 32-row tile of K/V live
// in shared memory; each thread owns up to ACC output accumulators (ACC the
// power of two at or above H*D/256; the slots past H*D stay idle).
#include "ds4c_internal.cuh"

namespace ds4c {
namespace {

constexpr int AT_THREADS = 256;
constexpr int AT_ROWS = 32;

struct RowSrc {
    const float *ring;   // this sequence's ring [S][D]
    const float *comp;   // this sequence's compressed rows [cap][D]
    const float *raw_new;
    uint64_t pos0;       // first position served by raw_new
    int64_t raw_row0;    // raw_new row of position pos0
};

template <int ACC>
__global__ void __launch_bounds__(AT_THREADS) attn_simt_kernel(AttnArgs a, DecodePos dp) {
    extern __shared__ float sm[];
    const int D = a.D, H = a.H;
    const int n = blockIdx.x;                       // query index
    const int seq = (a.n_seq == 1) ? 0 : n;
    const uint64_t t = (a.n_seq == 1) ? a.pos0 + (uint64_t)n : dp.pos[n];
    RowSrc src;
    src.ring = a.ring + (size_t)seq * a.S * D;
    src.comp = a.comp + (size_t)seq * a.comp_cap * D;
    src.raw_new = a.raw_new;
    src.pos0 = (a.n_seq == 1) ? a.pos0 : t;
    src.raw_row0 = (a.n_seq == 1) ? 0 : n;

    float *Qs = sm;                                 // [H][D]
    float *Xs = Qs + (size_t)H * D;                 // [AT_ROWS][D+1]
    float *Ps = Xs + (size_t)AT_ROWS * (D + 1);     // [H][AT_ROWS]
    float *m_run = Ps + (size_t)H * AT_ROWS;        // [H]
    float *l_run = m_run + H;                       // [H]
    float *alpha = l_run + H;                       // [H]
    int *clist = reinterpret_cast<int *>(alpha + H);  // [k] filtered compressed rows
    __shared__ int n_comp_sh;

    // Row set: raw positions [first, t], then compressed rows.
    const uint64_t first = (t + 1 > (uint64_t)a.S) ? t + 1 - (uint64_t)a.S : 0;
    const int n_raw = (int)(t - first + 1);
    int n_comp = 0;
    if (a.ratio == 4) {
        if (threadIdx.x == 0) {
            const uint64_t visible = (t + 1) / 4;
            const int32_t *tk = a.topk + (size_t)n * a.k;
            int c = 0;
            for (int i = 0; i < a.k; i++) {
                const int32_t idx = tk[i];
                if (idx < 0) continue;
                if ((uint64_t)idx >= visible) break;
                clist[c++] = idx;
            }
            n_comp_sh = c;
        }
        __syncthreads();
        n_comp = n_comp_sh;
    } else if (a.ratio == 128) {
        n_comp = (int)((t + 1) / 128);
    }
    const int n_rows = n_raw + n_comp;

    const float *q = a.q + (size_t)n * H * D;
    for (int e = threadIdx.x; e < H * D; e += AT_THREADS) Qs[e] = q[e];
    for (int h = threadIdx.x; h < H; h += AT_THREADS) { m_run[h] = -INFINITY; l_run[h] = 0.f; }

    float acc[ACC];
#pragma unroll
    for (int m = 0; m < ACC; m++) acc[m] = 0.f;

    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    for (int r0 = 0; r0 < n_rows; r0 += AT_ROWS) {
        __syncthreads();
        // stage rows r0 .. r0+31 (zeros past the end)
        for (int e = threadIdx.x; e < AT_ROWS * D; e += AT_THREADS) {
            const int r = e / D, col = e % D;
            const int i = r0 + r;
            float v = 0.f;
            if (i < n_raw) {
                const uint64_t p = first + (uint64_t)i;
                v = (p >= src.pos0) ? src.raw_new[(size_t)(src.raw_row0 + (int64_t)(p - src.pos0)) * D + col]
                                    : src.ring[(size_t)(p % (uint64_t)a.S) * D + col];
            } else if (i < n_rows) {
                const int c = (a.ratio == 4) ? clist[i - n_raw] : (i - n_raw);
                v = src.comp[(size_t)c * D + col];
            }
            Xs[r * (D + 1) + col] = v;
        }
        __syncthreads();
        // logits: lane = row, warps stride over heads
        {
            const int r = lane;
            const bool valid = (r0 + r) < n_rows;
            for (int h = warp; h < H; h += AT_THREADS / 32) {
                const float *qh = Qs + (size_t)h * D;
                const float *xr = Xs + r * (D + 1);
                float s = 0.f;
                for (int dd = 0; dd < D; dd++) s = fmaf(qh[dd], xr[dd], s);
                Ps[h * AT_ROWS + r] = valid ? s * a.scale : -INFINITY;
            }
        }
        __syncthreads();
        // online softmax bookkeeping, one warp per head
        for (int h = warp; h < H; h += AT_THREADS / 32) {
            const float s = Ps[h * AT_ROWS + lane];
            float mt = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            const float m_old = m_run[h];
            const float m_new = fmaxf(m_old, mt);
            const float p = expf(s - m_new);
            float ps = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            Ps[h * AT_ROWS + lane] = p;
            __syncwarp();
            if (lane == 0) {
                const float al = expf(m_old - m_new);   // 0 on the first tile
                alpha[h] = al;
                l_run[h] = l_run[h] * al + ps;
                m_run[h] = m_new;
            }
        }
        __syncthreads();
        // accumulate P X into this thread's outputs e = tid + 256*m
#pragma unroll
        for (int m = 0; m < ACC; m++) {
            const int e = threadIdx.x + AT_THREADS * m;
            if (e >= H * D) break;
            const int h = e / D, dd = e % D;
            float v = acc[m] * alpha[h];
            const float *ph = Ps + h * AT_ROWS;
#pragma unroll 8
            for (int r = 0; r < AT_ROWS; r++) v = fmaf(ph[r], Xs[r * (D + 1) + dd], v);
            acc[m] = v;
        }
    }
    __syncthreads();
    float *o = a.out + (size_t)n * H * D;
#pragma unroll
    for (int m = 0; m < ACC; m++) {
        const int e = threadIdx.x + AT_THREADS * m;
        if (e >= H * D) break;
        const int h = e / D;
        o[e] = acc[m] / l_run[h];
    }
}

template <int ACC>
cudaError_t launch_acc(const AttnArgs &a, const DecodePos &dp, int n_q, cudaStream_t s) {
    const size_t smem = sizeof(float) * ((size_t)a.H * a.D + (size_t)AT_ROWS * (a.D + 1) + (size_t)a.H * AT_ROWS +
                                         3 * (size_t)a.H) + sizeof(int) * (size_t)(a.k + 1);
    cudaError_t e = ensure_dyn_smem(attn_simt_kernel<ACC>, smem);
    if (e != cudaSuccess) return e;
    attn_simt_kernel<ACC><<<n_q, AT_THREADS, smem, s>>>(a, dp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnArgs &a, const DecodePos *p, cudaStream_t s) {
    const int n_q = a.n_seq * a.n_tok;
    if (n_q <= 0) return cudaSuccess;
    DecodePos dp{};
    if (a.n_seq > 1) dp = *p;
    int acc = 2;                                         // accumulators per thread: a power of two
    while (acc * AT_THREADS < a.H * a.D) acc *= 2;
    switch (acc) {
        case 2: return launch_acc<2>(a, dp, n_q, s);
        case 4: return launch_acc<4>(a, dp, n_q, s);
        case 8: return launch_acc<8>(a, dp, n_q, s);
        case 16: return launch_acc<16>(a, dp, n_q, s);
        case 32: return launch_acc<32>(a, dp, n_q, s);
        case 64: return launch_acc<64>(a, dp, n_q, s);
        case 128: return launch_acc<128>(a, dp, n_q, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ds4c
