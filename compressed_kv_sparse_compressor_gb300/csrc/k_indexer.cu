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
__device__ unsigned long long g_idx_wait_ns = kWaitNsDefault;

namespace {

// ---------------------------------------------------------------------------
// K4 prefill: n_tok queries of one sequence against every visible row.  128 x
// 128 (query x row) tile per 128-thread block, 8 queries x 16 rows per thread,
// d consumed in 16-wide slices in index order (so each output is exactly the
// in-order fmaf chain), slices double-buffered in shared memory, k-major.
// Shared-memory delivery (32 floats per clock per SM) against the FMA pipe
// (128 per clock) sets the register tile: 24 operands per 128 FMAs per k.  A
// thread's rows are tx*4 + 32g + (0..3), g < 4, so the eight threads of a
// quarter-warp read one 128-byte line of the row slice and share the query
// values.  The FMAs are packed (fma.rn.f32x2: two independent round-to-nearest
// fmas, one per lane half) over pairs of rows, which halves the issue slots
// the chain takes; each output is still its own in-order fmaf chain.  Tiles
// wholly past the visibility triangle are skipped.
// ---------------------------------------------------------------------------
constexpr int SB = 128, SK = 16, SP = SB + 4, ST = 128;

// 128 queries x 16 d and 128 rows x 16 d: 512 float4 each, 4 per thread
__device__ __forceinline__ void fetch_slice(float4 (&qv)[4], float4 (&rv)[4], const IndexerArgs &a, int j0, int c0,
                                            uint64_t vis_max, int i0) {
#pragma unroll
    for (int h = 0; h < 4; h++) {
        const int f = threadIdx.x + ST * h;
        const int r = f >> 2, k4 = (f & 3) * 4;
        const int j = j0 + r, c = c0 + r;
        qv[h] = make_float4(0.f, 0.f, 0.f, 0.f);
        rv[h] = qv[h];
        if (j < a.n_tok) qv[h] = *reinterpret_cast<const float4 *>(a.q + (size_t)j * a.d + i0 + k4);
        if ((uint64_t)c < vis_max) rv[h] = *reinterpret_cast<const float4 *>(a.rows + (size_t)c * a.d + i0 + k4);
    }
}
__device__ __forceinline__ void store_slice(float (*As)[SP], float (*Bs)[SP], const float4 (&qv)[4], const float4 (&rv)[4]) {
#pragma unroll
    for (int h = 0; h < 4; h++) {
        const int f = threadIdx.x + ST * h;
        const int r = f >> 2, k4 = (f & 3) * 4;
        As[k4 + 0][r] = qv[h].x; As[k4 + 1][r] = qv[h].y; As[k4 + 2][r] = qv[h].z; As[k4 + 3][r] = qv[h].w;
        Bs[k4 + 0][r] = rv[h].x; Bs[k4 + 1][r] = rv[h].y; Bs[k4 + 2][r] = rv[h].z; Bs[k4 + 3][r] = rv[h].w;
    }
}

// two floats as the halves of one 64-bit register pair, and back
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__global__ void __launch_bounds__(ST, 2) score_prefill_kernel(IndexerArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int j0 = blockIdx.y * SB, c0 = blockIdx.x * SB;
    const int jlast = min(j0 + SB, a.n_tok) - 1;
    const uint64_t vis_max = (a.pos0 + (uint64_t)jlast + 1) / 4;
    if ((uint64_t)c0 >= vis_max) return;
    __shared__ __align__(16) float As[2][SK][SP];
    __shared__ __align__(16) float Bs[2][SK][SP];
    const int tx = threadIdx.x % 8, ty = threadIdx.x / 8;
    uint64_t acc2[8][8];          // rows (2m, 2m+1) of query i, one packed pair
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int m = 0; m < 8; m++) acc2[i][m] = 0ull;
    float4 qv[4], rv[4];
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
            uint64_t rr[8];
#pragma unroll
            for (int g = 0; g < 4; g++) {
                const float4 b = *reinterpret_cast<const float4 *>(&Bs[cur][kk][32 * g + tx * 4]);
                rr[2 * g] = pack2(b.x, b.y);
                rr[2 * g + 1] = pack2(b.z, b.w);
            }
            const float qa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint64_t qq = pack2(qa[i], qa[i]);
#pragma unroll
                for (int m = 0; m < 8; m++) asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i][m]) : "l"(qq), "l"(rr[m]));
            }
        }
        if (sl + 1 < nslices) store_slice(As[cur ^ 1], Bs[cur ^ 1], qv, rv);
        __syncthreads();
    }
    float acc[8][16];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int m = 0; m < 8; m++) unpack2(acc2[i][m], acc[i][2 * m], acc[i][2 * m + 1]);
    const bool vec = (a.lds % 4) == 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        const int j = j0 + ty * 8 + i;
        if (j >= a.n_tok) continue;
        const uint64_t vis = (a.pos0 + (uint64_t)j + 1) / 4;
        float *dst = a.scores + (size_t)j * a.lds;
#pragma unroll
        for (int g = 0; g < 4; g++) {
            const int cb = c0 + 32 * g + tx * 4;
            if (vec && (uint64_t)cb + 4 <= vis) {
                *reinterpret_cast<float4 *>(dst + cb) =
                    make_float4(acc[i][4 * g], acc[i][4 * g + 1], acc[i][4 * g + 2], acc[i][4 * g + 3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; e++)
                    if ((uint64_t)(cb + e) < vis) dst[cb + e] = acc[i][4 * g + e];
            }
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
    pdl_wait();
    pdl_launch_dependents();
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
__device__ __forceinline__ uint32_t idx_smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// Bounded wait for the completion of phase `parity` of an mbarrier (the time is
// checked every 256 polls); false when limit_ns ran out first.
__device__ __forceinline__ bool idx_bounded_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 255u) == 255u) {
            uint64_t now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            if (t0 == 0) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
}

// Self-test of the error path: one thread waits on a barrier that nothing
// arrives on (bounded), raises the error word when the limit runs out.
__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    const uint32_t b = idx_smem_u32(&bar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(b) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!idx_bounded_wait(b, 0, limit_ns)) atomicOr(&g_idx_err, 2u);
    }
}

template <int DD>
__global__ void __launch_bounds__(128) score_decode_tma_kernel(const __grid_constant__ CUtensorMap rowsMap, IndexerArgs a,
                                                               DecodePos dp, int idx_cap, int early) {
    static_assert(DD % 32 == 0 && DD <= 128, "staged rows: d/32 boxes of 16 KB");
    constexpr int SEG = DD / 32;
    extern __shared__ uint8_t sm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bar;
    __shared__ float qs[DD];
    pdl_launch_dependents();
    const int b = blockIdx.y;
    const uint64_t vis = (dp.pos[b] + 1) / 4;
    const int c0 = blockIdx.x * 128;
    if ((uint64_t)c0 >= vis) {                          // no rows (early: as a block of old rows)
        if (!early) pdl_wait();
        return;
    }
    // early: the previous kernel is this step's decode compressor, which writes no row but the
    // newest.  Rows before the newest visible one were then written by earlier steps: a block
    // of only those scores them while the compressor still runs and exits without waiting.
    // The block holding a sequence's newest row, which this step may just have emitted, waits
    // first; every sequence with a visible row has one, so this grid still completes only
    // after the compressor (and the kernels after it see what the compressor wrote).
    const bool wait_first = !early || (uint64_t)c0 + 128 >= vis;
    if (wait_first) pdl_wait();
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
    // bounded wait for the boxes; a wait that gives up raises the error word and, before
    // the CTA returns, waits (bounded again) for the boxes still landing in its shared memory
    if (!idx_bounded_wait(bar_a, 0, g_idx_wait_ns)) {
        atomicOr(&g_idx_err, 1u);                       // every thread that gave up: its score is missing
        idx_bounded_wait(bar_a, 0, kDrainNs);
        return;
    }
    const int t = threadIdx.x;
    const int c = c0 + t;
    if ((uint64_t)c >= vis) return;                     // (only in the newest row's block, which has waited)
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
// K5 top-k, one CTA per query: the k largest scores among the visible rows,
// listed in ascending row order, equal scores going to the lower row.
//
// Keys are order-preserving u32 images of the scores.  Main path, two reads
// of the score row:
//   1. a 4096-bin histogram of the top 12 key bits (shared atomics); a suffix
//      scan over it gives the bin b* that holds the k-th largest key;
//   2. rows in bins above b* are selected outright (one bitmap word per 32
//      rows, from a warp ballot); rows in b* are copied to a candidate list;
//   3. two 1024-bin passes over the candidates resolve the low 20 bits: the
//      k-th largest key K* and how many rows equal to K* are taken;
//   4. candidates above K* join the bitmap, those equal to K* go to a second
//      bitmap, and one in-order scan of both writes the list, taking the
//      lowest rows of K* first.
// When b* holds more rows than the candidate list (heavy ties), the CTA runs
// a plain 4-bit radix select instead (private per-thread counters, 8 passes,
// then an ordered compaction).
// Prefill: 256 threads, the row stays in global memory (the second read hits
// L2), several CTAs per SM.  Decode: 1024 threads, the keys resident in shared
// memory.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t order_key(float s) {
    uint32_t u = __float_as_uint(s + 0.0f);          // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int TK_HBITS = 12;         // main path: bits of the first histogram
constexpr int TK_HBINS = 1 << TK_HBITS;
constexpr int TK_CAND = 2048;        // main path: candidate list (key, row)
constexpr int TK_BINS = 16;          // radix path: 4-bit digits
constexpr int TK_RCAND = 4096;       // radix path: survivors compacted once they fit
constexpr int TK_UNR = 16;           // independent score loads in flight per thread
constexpr int TK_PREFILL = 256, TK_DECODE = 1024;

// Dynamic shared memory in u32 words:
//   bins [max(4096, 16 T)] | candidate keys [2048] | candidate rows [2048] |
//   selected bitmap [wcap] | equal-key bitmap [wcap] | resident keys [vmax rounded up to 4]
// (wcap even, so that the resident keys start on 16 bytes and are stored four at a time)
// The radix path reuses the bins as its per-thread counters and the candidate
// lists as its 4096-key survivor buffer.
template <int T>
__host__ __device__ constexpr int tk_bin_words() { return TK_HBINS > TK_BINS * T ? TK_HBINS : TK_BINS * T; }
inline uint64_t tk_wcap(uint64_t vmax) { return ((vmax + 31) / 32 + 1) & ~(uint64_t)1; }
template <int T>
size_t tk_smem(uint64_t vmax, bool resident) {
    return sizeof(uint32_t) * ((size_t)tk_bin_words<T>() + 2 * TK_CAND + 2 * tk_wcap(vmax) +
                               (resident ? (vmax + 3) / 4 * 4 : 0));
}
static_assert(2 * TK_CAND >= TK_RCAND, "radix survivors fit the candidate lists");

// Suffix crossing over bins[0, nbins) (nbins a multiple of T, at least T),
// counted from the top bin down: the bin holding the need-th largest element
// (res[0]) and that element's rank inside the bin (res[1], 1 = the bin's
// largest).  Needs need >= 1 and at most the bins' total.  Ends on a barrier.
template <int T>
__device__ __forceinline__ void tk_crossing(const uint32_t *bins, int nbins, uint32_t need, uint32_t *warp_sum,
                                            uint32_t *res) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = nbins / T;
    const int hi = nbins - tid * per;                       // this thread's bins: [hi - per, hi)
    uint32_t local = 0;
    for (int b = hi - 1; b >= hi - per; b--) local += bins[b];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    for (int w = 0; w < warp; w++) incl += warp_sum[w];
    const uint32_t excl = incl - local;
    if (excl < need && incl >= need) {
        uint32_t r = need - excl;
        for (int b = hi - 1; b >= hi - per; b--) {
            const uint32_t h = bins[b];
            if (h >= r) {
                res[0] = (uint32_t)b;
                res[1] = r;
                break;
            }
            r -= h;
        }
    }
    __syncthreads();
}

// Radix path: 4 bits per pass from the top give K* and how many rows equal to
// K* to keep; once the keys that still match the resolved prefix fit the
// survivor buffer, later passes scan only those.  Then each warp owns a
// contiguous range of rows and one exchange of per-warp counts gives every
// warp its output offset.  cnt: [16][T] words, cand: [4096] words.
template <int T, typename KeyAt>
__device__ void tk_radix(int V, int k, int32_t *out, KeyAt key_at, uint32_t *cnt, uint32_t *cand) {
    constexpr int NW = T / 32;
    __shared__ uint32_t tot[TK_BINS];
    __shared__ uint32_t sh_prefix, sh_match, sh_ncand;
    __shared__ int sh_remaining, sh_compacted;
    __shared__ int sh_gt[NW], sh_eq[NW];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) { sh_prefix = 0; sh_remaining = k; sh_compacted = 0; sh_ncand = 0; }
    __syncthreads();
    for (int shift = 28; shift >= 0; shift -= 4) {
#pragma unroll
        for (int d = 0; d < TK_BINS; d++) cnt[d * T + tid] = 0;
        const uint32_t prefix = sh_prefix;
        const uint32_t hmask = (shift == 28) ? 0u : (0xffffffffu << (shift + 4));
        if (sh_compacted) {
            const int n = (int)sh_ncand;
            for (int i = tid; i < n; i += T) {
                const uint32_t key = cand[i];
                if ((key & hmask) == prefix) cnt[((key >> shift) & 15u) * T + tid] += 1u;
            }
        } else {
            for (int base = 0; base < V; base += T * TK_UNR) {
                uint32_t kv[TK_UNR];
#pragma unroll
                for (int u = 0; u < TK_UNR; u++) {
                    const int i = base + u * T + tid;
                    kv[u] = (i < V) ? key_at(i) : 0u;
                }
#pragma unroll
                for (int u = 0; u < TK_UNR; u++) {
                    const int i = base + u * T + tid;
                    if (i < V && (kv[u] & hmask) == prefix) cnt[((kv[u] >> shift) & 15u) * T + tid] += 1u;
                }
            }
        }
        __syncthreads();
        for (int bin = warp; bin < TK_BINS; bin += NW) {
            uint32_t v = 0;
            for (int j = lane; j < T; j += 32) v += cnt[bin * T + j];
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
        if (!sh_compacted && shift > 0 && sh_match <= (uint32_t)TK_RCAND) {
            const uint32_t np = sh_prefix, nm = 0xffffffffu << shift;
            for (int base = warp * 32; base < V; base += T) {
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
    const int per = ((V + NW - 1) / NW + 31) & ~31;
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
        if (sel && sel_run + __popc(selm & lt) < k) out[sel_run + __popc(selm & lt)] = c;
        eq_run += __popc(eqm);
        sel_run += __popc(selm);
    }
}

// One histogram pass over the candidate keys ckey[0, nc): bins of key bits
// [lo, lo + nbits) among the keys whose bits above them equal `match` (every
// key when `all`), then the crossing for the need-th largest (res[0] = bin,
// res[1] = rank in the bin).  Ends on a barrier.
template <int T>
__device__ __forceinline__ void tk_cand_pass(uint32_t *bins, const uint32_t *ckey, int nc, int nbits, int lo, bool all,
                                             uint32_t match, uint32_t need, uint32_t *warp_a, uint32_t *res) {
    const int nb = 1 << nbits;
    for (int i = threadIdx.x; i < nb; i += T) bins[i] = 0;
    __syncthreads();
    for (int j = threadIdx.x; j < nc; j += T) {
        const uint32_t key = ckey[j];
        if (all || (key >> (lo + nbits)) == match) atomicAdd(&bins[(key >> lo) & (uint32_t)(nb - 1)], 1u);
    }
    __syncthreads();
    tk_crossing<T>(bins, nb, need, warp_a, res);
}

// Candidates above K* join the selection bitmap, those equal to K* go to the
// equal-key bitmap.  Ends on a barrier.
template <int T>
__device__ __forceinline__ void tk_mark(const uint32_t *ckey, const uint32_t *crow, int nc, uint32_t kstar, uint32_t *sel,
                                        uint32_t *eqm) {
    for (int j = threadIdx.x; j < nc; j += T) {
        const uint32_t key = ckey[j], r = crow[j];
        if (key > kstar) atomicOr(&sel[r >> 5], 1u << (r & 31u));
        else if (key == kstar) atomicOr(&eqm[r >> 5], 1u << (r & 31u));
    }
    __syncthreads();
}

// The list in row order: the selected rows plus the first take_eq rows equal
// to K*.  Each thread owns a run of bitmap words; an exclusive scan of the
// per-thread counts gives its output offset and the equal-key rank.  No write
// lands past the k entries of the list, whatever the bitmaps hold.
template <int T>
__device__ __forceinline__ void tk_emit(const uint32_t *sel, const uint32_t *eqm, int W, uint32_t take_eq, int32_t *out,
                                        int k, uint32_t *warp_a, uint32_t *warp_b) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (W + T - 1) / T;
    const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
    uint32_t cs = 0, ce = 0;
    for (int w = w0; w < w1; w++) {
        cs += __popc(sel[w]);
        ce += __popc(eqm[w]);
    }
    uint32_t is = cs, ie = ce;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t vs = __shfl_up_sync(0xffffffffu, is, o), ve = __shfl_up_sync(0xffffffffu, ie, o);
        if (lane >= o) { is += vs; ie += ve; }
    }
    if (lane == 31) { warp_a[warp] = is; warp_b[warp] = ie; }
    __syncthreads();
    for (int w = 0; w < warp; w++) { is += warp_a[w]; ie += warp_b[w]; }
    uint32_t eq_before = ie - ce;
    uint32_t dst = (is - cs) + min(eq_before, take_eq);
    for (int w = w0; w < w1; w++) {
        const uint32_t e_all = eqm[w];
        uint32_t e = 0;
        if (eq_before < take_eq) {
            uint32_t want = take_eq - eq_before;
            uint32_t rest = e_all;
            while (rest && want) {                       // the lowest `want` equal rows of the word
                const uint32_t lb = rest & (0u - rest);
                e |= lb;
                rest ^= lb;
                want--;
            }
        }
        eq_before += __popc(e_all);
        uint32_t m = sel[w] | e;
        while (m) {
            if (dst < (uint32_t)k) out[dst] = w * 32 + (__ffs(m) - 1);
            dst++;
            m &= m - 1u;
        }
    }
}

// Query q: visible rows V = (pos + 1) / 4; fewer than k + 1 rows lists them all
// and pads with -1.
__device__ __forceinline__ bool tk_trivial(const IndexerArgs &a, int V, int32_t *out, int T) {
    if (V > a.k) return false;
    for (int i = threadIdx.x; i < a.k; i += T) out[i] = (i < V) ? i : -1;
    return true;
}

template <int T, bool RESIDENT>
__global__ void __launch_bounds__(T) topk_kernel(IndexerArgs a, DecodePos dp, int wcap) {
    constexpr int NW = T / 32;
    extern __shared__ uint32_t sm_tk[];
    uint32_t *bins = sm_tk;
    uint32_t *ckey = bins + tk_bin_words<T>();
    uint32_t *crow = ckey + TK_CAND;
    uint32_t *sel = crow + TK_CAND;
    uint32_t *eqm = sel + wcap;
    uint32_t *keys = eqm + wcap;                         // RESIDENT only
    __shared__ uint32_t warp_a[NW], warp_b[NW], res[2], sh_nc;
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // prefill takes the queries last first: the score rows written last are the
    // ones still in L2
    const int q = (a.n_seq == 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const uint64_t pos = (a.n_seq == 1) ? a.pos0 + (uint64_t)q : dp.pos[q];
    const int V = (int)((pos + 1) / 4);
    const int k = a.k;
    int32_t *out = a.topk + (size_t)q * k;
    if (tk_trivial(a, V, out, T)) return;
    const float *s = a.scores + (size_t)q * a.lds;
    const int W = (V + 31) / 32;
    for (int i = tid; i < TK_HBINS; i += T) bins[i] = 0;
    for (int i = tid; i < W; i += T) eqm[i] = 0;
    if (tid == 0) sh_nc = 0;
    __syncthreads();
    // 1. histogram of the top 12 key bits (resident: the keys land in shared memory).  A row
    //    of the workspace (16-byte aligned, a multiple of 4 floats long) is read four scores
    //    per load; its floats past V exist and are skipped (resident: stored as keys 0, never read).
    constexpr int SH1 = 32 - TK_HBITS;
    constexpr int U4 = TK_UNR / 4;
    const bool vec4 = (a.lds & 3) == 0 && (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
    const float4 *s4 = reinterpret_cast<const float4 *>(s);
    const int V4 = (V + 3) / 4;
    if (vec4) {
        for (int base = 0; base < V4; base += T * U4) {
            float4 v[U4];
#pragma unroll
            for (int u = 0; u < U4; u++) {
                const int i4 = base + u * T + tid;
                v[u] = (i4 < V4) ? (RESIDENT ? __ldcs(s4 + i4) : __ldg(s4 + i4)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U4; u++) {
                const int i4 = base + u * T + tid;
                const float e4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                uint32_t k4[4];
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    k4[e] = 4 * i4 + e < V ? order_key(e4[e]) : 0u;
                    if (4 * i4 + e < V) atomicAdd(&bins[k4[e] >> SH1], 1u);
                }
                if (RESIDENT && i4 < V4)
                    *reinterpret_cast<uint4 *>(keys + 4 * i4) = make_uint4(k4[0], k4[1], k4[2], k4[3]);
            }
        }
    } else
    for (int base = 0; base < V; base += T * TK_UNR) {
        float v[TK_UNR];
#pragma unroll
        for (int u = 0; u < TK_UNR; u++) {
            const int i = base + u * T + tid;
            v[u] = (i < V) ? (RESIDENT ? __ldcs(s + i) : __ldg(s + i)) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < TK_UNR; u++) {
            const int i = base + u * T + tid;
            if (i < V) {
                const uint32_t key = order_key(v[u]);
                if (RESIDENT) keys[i] = key;
                atomicAdd(&bins[key >> SH1], 1u);
            }
        }
    }
    __syncthreads();
    auto key_at = [&](int i) -> uint32_t { return RESIDENT ? keys[i] : order_key(__ldg(s + i)); };
    tk_crossing<T>(bins, TK_HBINS, (uint32_t)k, warp_a, res);
    const uint32_t bstar = res[0], rank1 = res[1];
    const int nc = (int)bins[bstar];
    if (nc > TK_CAND) {                                  // heavy ties in b*: plain radix select
        __syncthreads();
        tk_radix<T>(V, k, out, key_at, bins, ckey);
        return;
    }
    // 2. rows above b* are selected, rows in b* become candidates; a warp's 32
    //    rows are consecutive and 32-aligned, so its ballot is one bitmap word (four-score
    //    loads: a warp covers 128 rows, each lane a nibble of one of four words, which eight
    //    lanes OR together)
    if (vec4) {
        for (int base = 0; base < V4; base += T * U4) {
            float4 v[U4];
            uint4 kr[U4];
#pragma unroll
            for (int u = 0; u < U4; u++) {
                const int i4 = base + u * T + tid;
                if (RESIDENT) kr[u] = (i4 < V4) ? *reinterpret_cast<const uint4 *>(keys + 4 * i4) : make_uint4(0u, 0u, 0u, 0u);
                else v[u] = (i4 < V4) ? __ldcs(s4 + i4) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U4; u++) {
                const int g0 = base + u * T + warp * 32;     // the warp's first group of four rows
                if (4 * g0 >= V) continue;                   // the whole warp is past the end
                const int i4 = g0 + lane;
                uint32_t k4[4];
                if (RESIDENT) {
                    k4[0] = kr[u].x; k4[1] = kr[u].y; k4[2] = kr[u].z; k4[3] = kr[u].w;
                } else {
                    k4[0] = order_key(v[u].x); k4[1] = order_key(v[u].y); k4[2] = order_key(v[u].z);
                    k4[3] = order_key(v[u].w);
                }
                uint32_t nib = 0;
#pragma unroll
                for (int e = 0; e < 4; e++) {
                    const int r = 4 * i4 + e;
                    if (r >= V) continue;
                    const uint32_t key = k4[e];
                    const uint32_t b = key >> SH1;
                    if (b > bstar) nib |= 1u << e;
                    else if (b == bstar) {
                        const uint32_t o = atomicAdd(&sh_nc, 1u);
                        ckey[o] = key;
                        crow[o] = (uint32_t)r;
                    }
                }
                uint32_t x = nib << (4 * (lane & 7));
                x |= __shfl_xor_sync(0xffffffffu, x, 1);
                x |= __shfl_xor_sync(0xffffffffu, x, 2);
                x |= __shfl_xor_sync(0xffffffffu, x, 4);
                const int w = g0 / 8 + lane / 8;
                if ((lane & 7) == 0 && w < W) sel[w] = x;
            }
        }
    } else
    for (int base = 0; base < V; base += T * TK_UNR) {
        uint32_t kv[TK_UNR];
#pragma unroll
        for (int u = 0; u < TK_UNR; u++) {
            const int i = base + u * T + tid;
            kv[u] = (i < V) ? (RESIDENT ? keys[i] : order_key(__ldcs(s + i))) : 0u;
        }
#pragma unroll
        for (int u = 0; u < TK_UNR; u++) {
            const int row0 = base + u * T + warp * 32;
            if (row0 >= V) continue;                         // the whole warp is past the end
            const int i = row0 + lane;
            const bool in = i < V;
            const uint32_t b = kv[u] >> SH1;
            const unsigned above = __ballot_sync(0xffffffffu, in && b > bstar);
            const bool hit = in && b == bstar;
            const unsigned cm = __ballot_sync(0xffffffffu, hit);
            if (lane == 0) sel[row0 >> 5] = above;
            if (cm) {
                uint32_t off = 0;
                if (lane == 0) off = atomicAdd(&sh_nc, (uint32_t)__popc(cm));
                off = __shfl_sync(0xffffffffu, off, 0);
                if (hit) {
                    const uint32_t o = off + __popc(cm & ((1u << lane) - 1u));
                    ckey[o] = kv[u];
                    crow[o] = (uint32_t)i;
                }
            }
        }
    }
    __syncthreads();
    // 3. K*, the rank1-th largest candidate key (all in b*), and how many rows equal to it to
    //    take: bits 10..19 by a 1024-bin pass unless the candidates are few; then one warp
    //    ranks the (at most 32) candidates left, each lane counting the keys above and equal
    //    to its own; more than 32 left take the pass over bits 0..9
    uint32_t kstar, take_eq;                             // take_eq: rows equal to K*, lowest first
    uint32_t match = 0, need = rank1;                    // candidates whose key >> mshift == match
    int mshift = 32;                                     // (32: every candidate)
    if (nc > 32) {
        tk_cand_pass<T>(bins, ckey, nc, 10, 10, true, 0u, rank1, warp_a, res);
        const uint32_t b1 = res[0];
        need = res[1];
        match = (bstar << 10) | b1;
        mshift = 10;
    }
    const bool few = mshift == 32 || bins[match & 1023u] <= 32;
    __syncthreads();                                     // every thread has read the count before bins is reused
    if (few) {
        if (warp == 0) {
            // gather the matching candidates, one per lane, in candidate order
            uint32_t key = 0u;
            int cnt = 0;
            for (int j0 = 0; j0 < nc; j0 += 32) {
                const int j = j0 + lane;
                const uint32_t kj = j < nc ? ckey[j] : 0u;
                const bool mt = j < nc && (mshift == 32 || (kj >> mshift) == match);
                unsigned bm = __ballot_sync(0xffffffffu, mt);
                while (bm) {                             // at most 32 matches in all
                    const uint32_t v = __shfl_sync(0xffffffffu, kj, __ffs(bm) - 1);
                    if (lane == cnt) key = v;
                    cnt++;
                    bm &= bm - 1u;
                }
            }
            uint32_t gt = 0, eq = 0;
            for (int j = 0; j < cnt; j++) {
                const uint32_t o = __shfl_sync(0xffffffffu, key, j);
                gt += o > key ? 1u : 0u;
                eq += o == key ? 1u : 0u;
            }
            const unsigned m = __ballot_sync(0xffffffffu, lane < cnt && gt < need && need <= gt + eq);
            const int src = __ffs(m) - 1;
            const uint32_t kk = __shfl_sync(0xffffffffu, key, src), g = __shfl_sync(0xffffffffu, gt, src);
            if (lane == 0) {                             // (res may still be read: the pass's b1)
                warp_b[0] = kk;
                warp_b[1] = need - g;
            }
        }
        __syncthreads();
        kstar = warp_b[0];
        take_eq = warp_b[1];
    } else {
        tk_cand_pass<T>(bins, ckey, nc, 10, 0, false, match, need, warp_a, res);
        kstar = (match << 10) | res[0];
        take_eq = res[1];
    }
    // 4. candidates above K* join the selection, those equal to K* are marked apart
    tk_mark<T>(ckey, crow, nc, kstar, sel, eqm);
    // 5. in row order
    tk_emit<T>(sel, eqm, W, take_eq, out, k, warp_a, warp_b);
}

// Launch the top-k over n_q queries: the keys resident in shared memory when
// allowed and they fit, else read from the score rows each pass.  (At the
// largest index capacity the non-resident form needs 92 KB with 1024 threads.)
template <int T>
cudaError_t launch_topk(const IndexerArgs &a, const DecodePos &dp, int n_q, uint64_t vmax, bool allow_resident,
                        cudaStream_t s) {
    constexpr size_t LIMIT = 200 * 1024;
    if (vmax == 0) vmax = 1;
    const int wcap = (int)tk_wcap(vmax);
    cudaError_t e;
    if (allow_resident && tk_smem<T>(vmax, true) <= LIMIT) {
        const size_t smem = tk_smem<T>(vmax, true);
        if ((e = ensure_dyn_smem(topk_kernel<T, true>, smem)) != cudaSuccess) return e;
        e = launch_pdl(topk_kernel<T, true>, dim3(n_q), dim3(T), smem, s, a, dp, wcap);
    } else if (tk_smem<T>(vmax, false) <= LIMIT) {
        const size_t smem = tk_smem<T>(vmax, false);
        if ((e = ensure_dyn_smem(topk_kernel<T, false>, smem)) != cudaSuccess) return e;
        e = launch_pdl(topk_kernel<T, false>, dim3(n_q), dim3(T), smem, s, a, dp, wcap);
    } else {
        return cudaErrorNotSupported;
    }
    if (e == cudaSuccess) pdl_prev() = PdlPrev{s, PDL_TOPK};
    return e;
}


// ---------------------------------------------------------------------------
// Multi-head indexer score ("Metal グラフと圧縮 KV の実装を読む" §6: 64 indexer heads
// score each compressed row).  Per query and row: for each head j the in-order
// fp32 fma chain of its query vector with the row, clamped at zero, then the
// weighted head sum as one more in-order fma chain, s = fma(w[j], relu(dot_j), s)
// (this library's reading of the head combine).  A 128-thread block scores 128
// rows (one per thread, the row held in registers) for QB queries whose head
// vectors and weights sit in shared memory (read as broadcasts).  Prefill: QB
// consecutive queries of one sequence; decode: one query (its sequence) per block.
// ---------------------------------------------------------------------------
template <int DD, int QB>
__global__ void __launch_bounds__(128) score_heads_kernel(IndexerArgs a, const float *__restrict__ w, int heads,
                                                          DecodePos dp, int decode) {
    extern __shared__ __align__(16) float hsm[];
    float *qs = hsm;                                   // [QB][heads][DD]
    float *ws = hsm + (size_t)QB * heads * DD;         // [QB][heads]
    pdl_wait();
    pdl_launch_dependents();
    const int n_q = decode ? a.n_seq : a.n_tok;
    const int qb0 = blockIdx.y * QB;
    const int seq = decode ? qb0 : 0;
    uint64_t vis[QB];
    uint64_t vmax = 0;
#pragma unroll
    for (int k = 0; k < QB; k++) {
        const int n = qb0 + k;
        vis[k] = 0;
        if (n < n_q) vis[k] = decode ? (dp.pos[n] + 1) / 4 : (a.pos0 + (uint64_t)n + 1) / 4;
        vmax = vis[k] > vmax ? vis[k] : vmax;
    }
    const uint64_t c0 = (uint64_t)blockIdx.x * 128;
    if (c0 >= vmax) return;                            // block-uniform, before any barrier
    const int hd = heads * DD;
    for (int i = threadIdx.x; i < QB * hd; i += 128) {
        const int k = i / hd;
        qs[i] = (qb0 + k < n_q) ? a.q[(size_t)(qb0 + k) * hd + (i - k * hd)] : 0.f;
    }
    for (int i = threadIdx.x; i < QB * heads; i += 128) {
        const int k = i / heads;
        ws[i] = (qb0 + k < n_q) ? w[(size_t)(qb0 + k) * heads + (i - k * heads)] : 0.f;
    }
    __syncthreads();
    const uint64_t c = c0 + threadIdx.x;
    if (c >= vmax) return;
    const float4 *row = reinterpret_cast<const float4 *>(a.rows + (size_t)seq * a.seq_stride + (size_t)c * DD);
    float4 v[DD / 4];
#pragma unroll
    for (int i = 0; i < DD / 4; i++) v[i] = __ldg(row + i);
    float s[QB];
#pragma unroll
    for (int k = 0; k < QB; k++) s[k] = 0.f;
    for (int j = 0; j < heads; j++) {
        float acc[QB];
#pragma unroll
        for (int k = 0; k < QB; k++) acc[k] = 0.f;
#pragma unroll
        for (int i = 0; i < DD / 4; i++) {
#pragma unroll
            for (int k = 0; k < QB; k++) {
                const float4 q4 = *reinterpret_cast<const float4 *>(qs + ((size_t)k * heads + j) * DD + 4 * i);
                acc[k] = __fmaf_rn(q4.x, v[i].x, acc[k]);
                acc[k] = __fmaf_rn(q4.y, v[i].y, acc[k]);
                acc[k] = __fmaf_rn(q4.z, v[i].z, acc[k]);
                acc[k] = __fmaf_rn(q4.w, v[i].w, acc[k]);
            }
        }
#pragma unroll
        for (int k = 0; k < QB; k++) s[k] = __fmaf_rn(ws[k * heads + j], acc[k] > 0.f ? acc[k] : 0.f, s[k]);
    }
#pragma unroll
    for (int k = 0; k < QB; k++)
        if (qb0 + k < n_q && c < vis[k]) a.scores[(size_t)(qb0 + k) * a.lds + c] = s[k];
}

// Hadamard + FP4 round trip of n_vec vectors of 4G floats: G threads per vector.
template <int G>
__global__ void __launch_bounds__(128) qat_vectors_kernel(const float *__restrict__ in, float *__restrict__ out,
                                                          int64_t n_vec, float c) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t vec = (int64_t)blockIdx.x * (128 / G) + threadIdx.x / G;
    const int t = threadIdx.x % G;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec < n_vec) v = *reinterpret_cast<const float4 *>(in + vec * 4 * G + 4 * t);
    indexer_qat_group<G>(v, c);                        // every lane takes part in the shuffles
    if (vec < n_vec) *reinterpret_cast<float4 *>(out + vec * 4 * G + 4 * t) = v;
}

}  // namespace

cudaError_t launch_indexer_prefill(const IndexerArgs &a, cudaStream_t s) {
    const uint64_t vis_max = (a.pos0 + (uint64_t)a.n_tok) / 4;
    if (a.n_tok <= 0) return cudaSuccess;
    if (vis_max > 0) {
        dim3 grid((unsigned)((vis_max + SB - 1) / SB), (unsigned)((a.n_tok + SB - 1) / SB));
        cudaError_t e = launch_pdl(score_prefill_kernel, grid, dim3(ST), 0, s, a);
        if (e != cudaSuccess) return e;
    }
    DecodePos dp{};
    return launch_topk<TK_PREFILL>(a, dp, a.n_tok, vis_max, false, s);
}

cudaError_t launch_indexer_decode(const IndexerArgs &a, const DecodePos &p, cudaStream_t s) {
    uint64_t vis_max = 0;
    for (int b = 0; b < a.n_seq; b++) vis_max = ((p.pos[b] + 1) / 4 > vis_max) ? (p.pos[b] + 1) / 4 : vis_max;
    const int early = pdl_prev_is(s, PDL_DECODE_COMPRESS) ? 1 : 0;
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
        e = launch_pdl(score_decode_tma_kernel<dd>, grid, dim3(128), smem, s, rm, a, p, (int)idx_cap, early); \
        if (e != cudaSuccess) return e;                                                                      \
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
            case 64: e = launch_pdl(score_decode_kernel<64>, grid, dim3(128), 0, s, a, p); break;
            case 128: e = launch_pdl(score_decode_kernel<128>, grid, dim3(128), 0, s, a, p); break;
            case 256: e = launch_pdl(score_decode_kernel<256>, grid, dim3(128), 0, s, a, p); break;
            case 512: e = launch_pdl(score_decode_kernel<512>, grid, dim3(128), 0, s, a, p); break;
            default: return cudaErrorInvalidValue;
        }
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return launch_topk<TK_DECODE>(a, p, a.n_seq, vis_max, true, s);
}

cudaError_t launch_indexer_heads(const IndexerArgs &a, const float *w, int heads, const DecodePos *dp, cudaStream_t s) {
    const bool decode = dp != nullptr;
    const int n_q = decode ? a.n_seq : a.n_tok;
    if (n_q <= 0) return cudaSuccess;
    uint64_t vis_max = 0;
    if (decode) {
        for (int b = 0; b < a.n_seq; b++) vis_max = ((dp->pos[b] + 1) / 4 > vis_max) ? (dp->pos[b] + 1) / 4 : vis_max;
    } else {
        vis_max = (a.pos0 + (uint64_t)a.n_tok) / 4;
    }
    DecodePos none{};
    const DecodePos &p = decode ? *dp : none;
    if (vis_max > 0) {
        const int QB = decode ? 1 : 4;
        const dim3 grid((unsigned)((vis_max + 127) / 128), (unsigned)((n_q + QB - 1) / QB));
        const size_t smem = (size_t)QB * heads * a.d * 4 + (size_t)QB * heads * 4;
        cudaError_t e = cudaErrorInvalidValue;
#define DS4C_HEADS(dd, qb)                                                                              \
        if (a.d == dd && QB == qb) {                                                                   \
            e = ensure_dyn_smem(score_heads_kernel<dd, qb>, smem);                                     \
            if (e == cudaSuccess)                                                                      \
                e = launch_pdl(score_heads_kernel<dd, qb>, grid, dim3(128), smem, s, a, w, heads, p, decode ? 1 : 0); \
        }
        DS4C_HEADS(64, 1)
        DS4C_HEADS(64, 4)
        DS4C_HEADS(128, 1)
        DS4C_HEADS(128, 4)
#undef DS4C_HEADS
        if (e != cudaSuccess) return e;
    }
    return decode ? launch_topk<TK_DECODE>(a, p, n_q, vis_max, true, s)
                  : launch_topk<TK_PREFILL>(a, p, n_q, vis_max, false, s);
}

cudaError_t launch_qat_vectors(const float *in, float *out, int64_t n_vec, int d, float c, cudaStream_t s) {
    if (n_vec <= 0) return cudaSuccess;
    const int G = d / 4;
    const int64_t blocks = (n_vec * G + 127) / 128;
    if (G == 16) return launch_pdl(qat_vectors_kernel<16>, dim3((unsigned)blocks), dim3(128), 0, s, in, out, n_vec, c);
    if (G == 32) return launch_pdl(qat_vectors_kernel<32>, dim3((unsigned)blocks), dim3(128), 0, s, in, out, n_vec, c);
    return cudaErrorInvalidValue;
}

cudaError_t idx_set_wait_ns(unsigned long long ns) { return cudaMemcpyToSymbol(g_idx_wait_ns, &ns, sizeof ns); }

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

unsigned int idx_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_idx_err, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_idx_err, &z, sizeof z);
    return v;
}

}  // namespace ds4c
