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
// the keys re-read from the score row each pass), then an ordered compaction that emits the
// selected indices in ascending order, ties at the threshold broken toward
// the lower index.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ds4c_internal.cuh"

namespace ds4c {

__device__ unsigned int g_idx_err;

namespace {

// ---------------------------------------------------------------------------
// K4 prefill: n_tok queries of one sequence against every visible row.  128 x
// 128 (query x row) tile per 256-thread block, 8 x 8 outputs per thread, d
// consumed in 16-wide slices in index order (so each output is exactly the
// in-order fmaf chain), slices double-buffered in shared memory (k-major, so
// a thread reads its 8 queries / 8 rows of one k as two 16-byte loads).
// Tiles wholly past the visibility triangle are skipped.
// ---------------------------------------------------------------------------
constexpr int SB = 128, SK = 16, SP = SB + 4;

// 128 rows x 16 k of q and of the index rows: 512 float4 each, 2 per thread
__device__ __forceinline__ void fetch_slice(float4 (&qv)[2], float4 (&rv)[2], const IndexerArgs &a, int j0, int c0,
                                            uint64_t vis_max, int i0) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int f = threadIdx.x + 256 * h;
        const int r = f >> 2, k4 = (f & 3) * 4;
        const int j = j0 + r, c = c0 + r;
        qv[h] = make_float4(0.f, 0.f, 0.f, 0.f);
        rv[h] = qv[h];
        if (j < a.n_tok) qv[h] = *reinterpret_cast<const float4 *>(a.q + (size_t)j * a.d + i0 + k4);
        if ((uint64_t)c < vis_max) rv[h] = *reinterpret_cast<const float4 *>(a.rows + (size_t)c * a.d + i0 + k4);
    }
}
__device__ __forceinline__ void store_slice(float (*As)[SP], float (*Bs)[SP], const float4 (&qv)[2], const float4 (&rv)[2]) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
        const int f = threadIdx.x + 256 * h;
        const int r = f >> 2, k4 = (f & 3) * 4;
        As[k4 + 0][r] = qv[h].x; As[k4 + 1][r] = qv[h].y; As[k4 + 2][r] = qv[h].z; As[k4 + 3][r] = qv[h].w;
        Bs[k4 + 0][r] = rv[h].x; Bs[k4 + 1][r] = rv[h].y; Bs[k4 + 2][r] = rv[h].z; Bs[k4 + 3][r] = rv[h].w;
    }
}

__global__ void __launch_bounds__(256, 2) score_prefill_kernel(IndexerArgs a) {
    const int j0 = blockIdx.y * SB, c0 = blockIdx.x * SB;
    const int jlast = min(j0 + SB, a.n_tok) - 1;
    const uint64_t vis_max = (a.pos0 + (uint64_t)jlast + 1) / 4;
    if ((uint64_t)c0 >= vis_max) return;
    __shared__ __align__(16) float As[2][SK][SP];
    __shared__ __align__(16) float Bs[2][SK][SP];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int k = 0; k < 8; k++) acc[i][k] = 0.f;
    float4 qv[2], rv[2];
    fetch_slice(qv, rv, a, j0, c0, vis_max, 0);
    store_slice(As[0], Bs[0], qv, rv);
    __syncthreads();
    const int nslices = a.d / SK;
    for (int sl = 0; sl < nslices; sl++) {
        const int cur = sl & 1;
        if (sl + 1 < nslices) fetch_slice(qv, rv, a, j0, c0, vis_max, (sl + 1) * SK);   // in flight during the FMAs
#pragma unroll
        for (int kk = 0; kk < SK; kk++) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[cur][kk][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[cur][kk][ty * 8 + 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][tx * 8]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[cur][kk][tx * 8 + 4]);
            const float qa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float rb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int k = 0; k < 8; k++) acc[i][k] = __fmaf_rn(qa[i], rb[k], acc[i][k]);
        }
        if (sl + 1 < nslices) store_slice(As[cur ^ 1], Bs[cur ^ 1], qv, rv);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int j = j0 + ty * 8 + i;
        if (j >= a.n_tok) continue;
        const uint64_t vis = (a.pos0 + (uint64_t)j + 1) / 4;
        float *dst = a.scores + (size_t)j * a.lds;
        const int cb = c0 + tx * 8;
        if ((uint64_t)cb + 8 <= vis && (a.lds % 4) == 0) {
            *reinterpret_cast<float4 *>(dst + cb) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            *reinterpret_cast<float4 *>(dst + cb + 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; k++)
                if ((uint64_t)(cb + k) < vis) dst[cb + k] = acc[i][k];
        }
    }
}

// ---------------------------------------------------------------------------
// K4 decode: one query per sequence; a 128-thread block scores 128 rows of
// its sequence, one row per thread: the thread loads its whole row (d floats)
// with independent 16-byte loads, then runs the in-order fma chain against q
// (broadcast from shared memory).
// ---------------------------------------------------------------------------
template <int DD>
__global__ void __launch_bounds__(128) score_decode_kernel(IndexerArgs a, DecodePos dp) {
    __shared__ float qs[DD];
    const int b = blockIdx.y;
    const uint64_t vis = (dp.pos[b] + 1) / 4;
    const int c = blockIdx.x * 128 + threadIdx.x;
    if ((uint64_t)(blockIdx.x * 128) >= vis) return;
    for (int i = threadIdx.x; i < DD; i += 128) qs[i] = a.q[(size_t)b * DD + i];
    __syncthreads();
    if ((uint64_t)c >= vis) return;
    const float4 *row = reinterpret_cast<const float4 *>(a.rows + (size_t)b * a.seq_stride + (size_t)c * DD);
    float4 v[DD / 4];
    // issue every load of the row before the first use (volatile keeps the order)
#pragma unroll
    for (int i = 0; i < DD / 4; i++)
        asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(v[i].x), "=f"(v[i].y), "=f"(v[i].z), "=f"(v[i].w)
                     : "l"(row + i));
    asm volatile("" ::: "memory");   // the q reads below stay after the row loads
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < DD / 4; i++) {
        s = __fmaf_rn(qs[4 * i + 0], v[i].x, s);
        s = __fmaf_rn(qs[4 * i + 1], v[i].y, s);
        s = __fmaf_rn(qs[4 * i + 2], v[i].z, s);
        s = __fmaf_rn(qs[4 * i + 3], v[i].w, s);
    }
    a.scores[(size_t)b * a.lds + c] = s;
}

// ---------------------------------------------------------------------------
// K4 decode, staged form (d <= 128): a 128-thread block scores 128 rows of its
// sequence.  The rows arrive in shared memory by TMA as d/32 boxes of [128
// rows][32 floats] in the 128-byte swizzle, so that thread t reads its own row
// (16-byte chunk j of row t sits at chunk j ^ (t & 7)) without bank conflicts;
// then the same in-order fma chain.  Several blocks share an SM, so the HBM
// stream has many boxes in flight.
// ---------------------------------------------------------------------------
constexpr unsigned long long IDX_WAIT_NS = 4000000000ull;

__device__ __forceinline__ uint32_t idx_smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

template <int DD>
__global__ void __launch_bounds__(128) score_decode_tma_kernel(const __grid_constant__ CUtensorMap rowsMap, IndexerArgs a,
                                                               DecodePos dp, int idx_cap) {
    static_assert(DD % 32 == 0 && DD <= 128, "staged rows: d/32 boxes of 16 KB");
    constexpr int SEG = DD / 32;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ float qs[DD];
    const int b = blockIdx.y;
    const uint64_t vis = (dp.pos[b] + 1) / 4;
    const int c0 = blockIdx.x * 128;
    if ((uint64_t)c0 >= vis) return;
    const uint32_t bar_a = idx_smem_u32(&bar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_a) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar_a), "r"(SEG * 128 * 128) : "memory");
        const int y = b * idx_cap + c0;
#pragma unroll
        for (int sg = 0; sg < SEG; sg++)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                    idx_smem_u32(sm + sg * 16384)),
                "l"(reinterpret_cast<uint64_t>(&rowsMap)), "r"(32 * sg), "r"(y), "r"(bar_a)
                : "memory");
    }
    for (int i = threadIdx.x; i < DD; i += 128) qs[i] = a.q[(size_t)b * DD + i];
    __syncthreads();
    // bounded wait for the boxes; a wait that gives up raises the error word
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar_a)
            : "memory");
        if (done) break;
        if ((it & 255u) == 255u) {
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (t0 == 0) t0 = now;
            else if (now - t0 > IDX_WAIT_NS) {
                atomicOr(&g_idx_err, 1u);
                return;
            }
        }
    }
    const int t = threadIdx.x;
    const int c = c0 + t;
    if ((uint64_t)c >= vis) return;
    float4 v[DD / 4];
#pragma unroll
    for (int sg = 0; sg < SEG; sg++)
#pragma unroll
        for (int j = 0; j < 8; j++)
            v[sg * 8 + j] = *reinterpret_cast<const float4 *>(sm + sg * 16384 + t * 128 + ((j ^ (t & 7)) * 16));
    float sc = 0.f;
#pragma unroll
    for (int i = 0; i < DD / 4; i++) {
        sc = __fmaf_rn(qs[4 * i + 0], v[i].x, sc);
        sc = __fmaf_rn(qs[4 * i + 1], v[i].y, sc);
        sc = __fmaf_rn(qs[4 * i + 2], v[i].z, sc);
        sc = __fmaf_rn(qs[4 * i + 3], v[i].w, sc);
    }
    a.scores[(size_t)b * a.lds + c] = sc;
}

PFN_cuTensorMapEncodeTiled_v12000 idx_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// ---------------------------------------------------------------------------
// K5 top-k, one CTA per query, in two forms.  Prefill (thousands of queries):
// 256 threads, the scores stay in global memory (each pass re-reads the row:
// the first read comes from HBM, the later ones hit L2), so a CTA holds only
// its counters and candidate buffer (32 KB) and several CTAs share an SM,
// hiding each other's barrier and scan latencies.  Decode (one query per
// sequence, a few dozen CTAs): 1024 threads with the row's keys resident in
// shared memory, so each pass is short.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s + 0.0f);          // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int TK_BINS = 16;          // 4-bit radix digits, 8 passes
constexpr int TK_CAND = 4096;        // survivors are compacted once they fit here
constexpr int TK_UNR = 4;            // independent score loads in flight per thread
// dynamic shared memory: counters [16][threads] | candidates [4096] | (resident keys [V])
template <int TK_THREADS>
constexpr size_t tk_fixed_smem() { return sizeof(uint32_t) * (TK_BINS * TK_THREADS + TK_CAND); }
constexpr int TK_PREFILL = 256, TK_DECODE = 1024;

template <int TK_THREADS, bool RESIDENT>
__global__ void __launch_bounds__(TK_THREADS) topk_kernel(IndexerArgs a, DecodePos dp) {
    constexpr int TK_WARPS = TK_THREADS / 32;
    extern __shared__ uint32_t sm_tk[];
    uint32_t *cnt = sm_tk;                              // cnt[bin * threads + tid], private per thread
    uint32_t *cand = sm_tk + TK_BINS * TK_THREADS;
    uint32_t *keys = cand + TK_CAND;                    // RESIDENT only
    __shared__ uint32_t tot[TK_BINS];
    __shared__ uint32_t sh_prefix, sh_match, sh_ncand;
    __shared__ int sh_remaining, sh_compacted;
    __shared__ int sh_gt[TK_WARPS], sh_eq[TK_WARPS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q = blockIdx.x;
    const uint64_t pos = (a.n_seq == 1) ? a.pos0 + (uint64_t)q : dp.pos[q];
    const int V = (int)((pos + 1) / 4);
    const int k = a.k;
    int32_t *out = a.topk + (size_t)q * k;
    if (V <= k) {
        for (int i = tid; i < k; i += TK_THREADS) out[i] = (i < V) ? i : -1;
        return;
    }
    const float *s = a.scores + (size_t)q * a.lds;
    if (RESIDENT) {
        for (int base = 0; base < V; base += TK_THREADS * TK_UNR) {
            float v[TK_UNR];
#pragma unroll
            for (int u = 0; u < TK_UNR; u++) {
                const int i = base + u * TK_THREADS + tid;
                if (i < V) v[u] = __ldcs(s + i);
            }
#pragma unroll
            for (int u = 0; u < TK_UNR; u++) {
                const int i = base + u * TK_THREADS + tid;
                if (i < V) keys[i] = order_key(v[u]);
            }
        }
    }
    // key of visible row i
    auto key_at = [&](int i) -> uint32_t { return RESIDENT ? keys[i] : order_key(__ldg(s + i)); };
    if (tid == 0) { sh_prefix = 0; sh_remaining = k; sh_compacted = 0; sh_ncand = 0; }
    __syncthreads();
    // Radix select, 4 bits per pass from the top: the key K* of the k-th largest
    // element and how many elements equal to K* to keep.  Counters are private
    // to each thread (no atomics); once the keys that still match the resolved
    // prefix fit in the candidate buffer, later passes scan only those.
    for (int shift = 28; shift >= 0; shift -= 4) {
#pragma unroll
        for (int d = 0; d < TK_BINS; d++) cnt[d * TK_THREADS + tid] = 0;
        const uint32_t prefix = sh_prefix;
        const uint32_t hmask = (shift == 28) ? 0u : (0xffffffffu << (shift + 4));
        if (sh_compacted) {
            const int n = (int)sh_ncand;
            for (int i = tid; i < n; i += TK_THREADS) {
                const uint32_t key = cand[i];
                if ((key & hmask) == prefix) cnt[((key >> shift) & 15u) * TK_THREADS + tid] += 1u;
            }
        } else {
            for (int base = 0; base < V; base += TK_THREADS * TK_UNR) {
                uint32_t kv[TK_UNR];
#pragma unroll
                for (int u = 0; u < TK_UNR; u++) {
                    const int i = base + u * TK_THREADS + tid;
                    kv[u] = (i < V) ? key_at(i) : 0u;
                }
#pragma unroll
                for (int u = 0; u < TK_UNR; u++) {
                    const int i = base + u * TK_THREADS + tid;
                    if (i < V && (kv[u] & hmask) == prefix) cnt[((kv[u] >> shift) & 15u) * TK_THREADS + tid] += 1u;
                }
            }
        }
        __syncthreads();
        for (int bin = warp; bin < TK_BINS; bin += TK_WARPS) {
            uint32_t v = 0;
            for (int j = lane; j < TK_THREADS; j += 32) v += cnt[bin * TK_THREADS + j];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) tot[bin] = v;
        }
        __syncthreads();
        if (tid == 0) {
            int rem = sh_remaining;
            int bin = TK_BINS - 1;
            for (; bin > 0; bin--) {
                const int h = (int)tot[bin];
                if (h >= rem) break;
                rem -= h;
            }
            sh_prefix = prefix | ((uint32_t)bin << shift);
            sh_remaining = rem;
            sh_match = tot[bin];
        }
        __syncthreads();
        if (!sh_compacted && shift > 0 && sh_match <= (uint32_t)TK_CAND) {
            // collect the keys that match the prefix resolved so far
            const uint32_t np = sh_prefix, nm = 0xffffffffu << shift;
            for (int base = warp * 32; base < V; base += TK_THREADS) {
                const int c = base + lane;
                const uint32_t key = (c < V) ? key_at(c) : 0u;
                const bool hit = c < V && (key & nm) == np;
                const unsigned m = __ballot_sync(0xffffffffu, hit);
                uint32_t off = 0;
                if (lane == 0 && m) off = atomicAdd(&sh_ncand, (uint32_t)__popc(m));
                off = __shfl_sync(0xffffffffu, off, 0);
                if (hit) cand[off + __popc(m & ((1u << lane) - 1u))] = key;
            }
            __syncthreads();
            if (tid == 0) sh_compacted = 1;
            __syncthreads();
        }
    }
    const uint32_t kstar = sh_prefix;
    const int remaining = sh_remaining;
    // Ordered selection: keep key > K*, and the first `remaining` (by index) of
    // key == K*.  Each warp owns a contiguous range of indices; one exchange of
    // per-warp counts gives every warp its output offset.
    const int per = ((V + TK_WARPS - 1) / TK_WARPS + 31) & ~31;
    const int w0 = warp * per, w1 = min(V, w0 + per);
    int gt_w = 0, eq_w = 0;
    for (int base = w0; base < w1; base += 32) {
        const int c = base + lane;
        const uint32_t key = (c < w1) ? key_at(c) : 0u;
        gt_w += __popc(__ballot_sync(0xffffffffu, c < w1 && key > kstar));
        eq_w += __popc(__ballot_sync(0xffffffffu, c < w1 && key == kstar));
    }
    if (lane == 0) { sh_gt[warp] = gt_w; sh_eq[warp] = eq_w; }
    __syncthreads();
    int eq_run = 0, sel_run = 0;
    for (int w = 0; w < warp; w++) {
        const int take = max(0, min(sh_eq[w], remaining - eq_run));
        sel_run += sh_gt[w] + take;
        eq_run += sh_eq[w];
    }
    const unsigned lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int c = base + lane;
        const uint32_t key = (c < w1) ? key_at(c) : 0u;
        const bool gt = c < w1 && key > kstar;
        const bool eq = c < w1 && key == kstar;
        const unsigned eqm = __ballot_sync(0xffffffffu, eq);
        const int eq_rank = eq_run + __popc(eqm & lt);
        const bool sel = gt || (eq && eq_rank < remaining);
        const unsigned selm = __ballot_sync(0xffffffffu, sel);
        if (sel) out[sel_run + __popc(selm & lt)] = c;
        eq_run += __popc(eqm);
        sel_run += __popc(selm);
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
    constexpr size_t smem = tk_fixed_smem<TK_PREFILL>();
    cudaError_t e = ensure_dyn_smem(topk_kernel<TK_PREFILL, false>, smem);
    if (e != cudaSuccess) return e;
    DecodePos dp{};
    topk_kernel<TK_PREFILL, false><<<a.n_tok, TK_PREFILL, smem, s>>>(a, dp);
    return cudaGetLastError();
}

cudaError_t launch_indexer_decode(const IndexerArgs &a, const DecodePos &p, cudaStream_t s) {
    uint64_t vis_max = 0;
    for (int b = 0; b < a.n_seq; b++) vis_max = ((p.pos[b] + 1) / 4 > vis_max) ? (p.pos[b] + 1) / 4 : vis_max;
    cudaError_t e;
    // staged rows by TMA when the row width allows it (d = 32, 64, 96 or 128)
    const int64_t idx_cap = a.d > 0 ? a.seq_stride / a.d : 0;
    bool staged = vis_max > 0 && a.d <= 128 && a.d % 32 == 0 && (reinterpret_cast<uintptr_t>(a.rows) & 15u) == 0 &&
                  idx_cap * a.d == a.seq_stride;
    CUtensorMap rm;
    if (staged) {
        auto fn = idx_encode_fn();
        cuuint64_t dims[2] = {(cuuint64_t)a.d, (cuuint64_t)((uint64_t)a.n_seq * (uint64_t)idx_cap)};
        cuuint64_t strides[1] = {(cuuint64_t)a.d * 4};
        cuuint32_t box[2] = {32, 128};
        cuuint32_t estr[2] = {1, 1};
        staged = fn && fn(&rm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(a.rows), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    if (staged) {
        dim3 grid((unsigned)((vis_max + 127) / 128), (unsigned)a.n_seq);
        const size_t smem = (size_t)(a.d / 32) * 16384 + 1024;
#define DS4C_SCORE_TMA(dd)                                                                                   \
    case dd:                                                                                                 \
        e = ensure_dyn_smem(score_decode_tma_kernel<dd>, smem);                                              \
        if (e != cudaSuccess) return e;                                                                      \
        score_decode_tma_kernel<dd><<<grid, 128, smem, s>>>(rm, a, p, (int)idx_cap);                          \
        break;
        switch (a.d) {
            DS4C_SCORE_TMA(32)
            DS4C_SCORE_TMA(64)
            DS4C_SCORE_TMA(96)
            DS4C_SCORE_TMA(128)
            default: return cudaErrorInvalidValue;
        }
#undef DS4C_SCORE_TMA
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else if (vis_max > 0) {
        dim3 grid((unsigned)((vis_max + 127) / 128), (unsigned)a.n_seq);
        switch (a.d) {
            case 64: score_decode_kernel<64><<<grid, 128, 0, s>>>(a, p); break;
            case 128: score_decode_kernel<128><<<grid, 128, 0, s>>>(a, p); break;
            case 256: score_decode_kernel<256><<<grid, 128, 0, s>>>(a, p); break;
            case 512: score_decode_kernel<512><<<grid, 128, 0, s>>>(a, p); break;
            default: return cudaErrorInvalidValue;
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = tk_fixed_smem<TK_DECODE>() + sizeof(uint32_t) * (size_t)(vis_max > 0 ? vis_max : 1);
    if (smem <= (size_t)200 * 1024) {
        e = ensure_dyn_smem(topk_kernel<TK_DECODE, true>, smem);
        if (e != cudaSuccess) return e;
        topk_kernel<TK_DECODE, true><<<a.n_seq, TK_DECODE, smem, s>>>(a, p);
    } else {            // the keys do not fit: read them from the score rows each pass
        e = ensure_dyn_smem(topk_kernel<TK_DECODE, false>, tk_fixed_smem<TK_DECODE>());
        if (e != cudaSuccess) return e;
        topk_kernel<TK_DECODE, false><<<a.n_seq, TK_DECODE, tk_fixed_smem<TK_DECODE>(), s>>>(a, p);
    }
    return cudaGetLastError();
}

unsigned int idx_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_idx_err, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_idx_err, &z, sizeof z);
    return v;
}

}  // namespace ds4c
