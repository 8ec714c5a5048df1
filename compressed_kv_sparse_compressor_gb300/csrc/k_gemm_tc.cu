// Projection GEMM on the 5th-generation tensor cores (K1):
//   C[g][m][n] = sum_k A[m][k] * B_g[n][k]   (bf16 operands, fp32 accumulate)
// for the wkv / wgate matrices of the attention and indexer lanes
// ("Metal グラフと圧縮 KV の実装を読む" §4-§5: both projections are coff*head_dim
// wide; all four share the hidden rows A, so one persistent launch covers them).
//
// Design (sm_103a):
//   - 128 x 256 output tile per CTA, K consumed in 64-element (128-byte) slices;
//     A and B slices arrive by TMA (cp.async.bulk.tensor, 128-byte swizzle) into
//     a 4-stage shared-memory ring guarded by mbarriers.
//   - One elected thread issues tcgen05.mma (kind::f16, M=128, N=256, K=16) with
//     the accumulator in tensor memory; two 256-column accumulators let the
//     epilogue of one tile overlap the main loop of the next.
//   - Warp roles: warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner),
//     warps 2-5 epilogue (tcgen05.ld 32x32b -> registers -> global fp32).
//   - Persistent grid of one CTA per SM over (group, n-tile, m-tile).
//   - Every mbarrier wait is bounded (4 s of %globaltimer); a wait that gives up
//     raises the library's device error word and the CTA winds down, freeing
//     its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "ds4c_internal.cuh"

namespace ds4c {

__device__ unsigned int g_gemm_tc_err;
__device__ unsigned long long g_gemm_wait_ns = kWaitNsDefault;

namespace {

constexpr int BM = 128, BK = 64;
constexpr int THREADS = 192;

// Tile width BN: 256 for prefill chunks; 32 for decode-sized M, where the
// weights are the traffic and more, narrower tiles spread them over the SMs.
// AR: A rows a stage holds.  BM for prefill; 32 for M <= 32 ("thin" stages of
// 8 KB, so twice as many stages are in flight): the M = 128 MMA then reads rows
// 32..127 of A from whatever follows the stage -- finite or not, they only feed
// accumulator rows that are never stored -- and a pad after the last stage keeps
// those reads inside the allocation.
template <int BN, int AR = BM>
struct GT {
    static constexpr int A_BYTES = AR * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = AR < BM ? (BN >= 128 ? 8 : 20) : (BN >= 128 ? 4 : 8);
    static constexpr int PAD = (BM - AR) * BK * 2;
    static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
    // barriers (2 * STAGES + 5) and the TMEM slot / abort flag after the stages, plus the
    // realignment of the base to 1024 bytes
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + PAD + 1024 + 8 * (2 * STAGES + 5) + 16;
    // instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major, M = 128, N = BN
    static constexpr uint32_t IDESC =
        (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
};

struct TcParams {
    int M, K;
    int m_tiles;
    int n_groups;
    int ksplit;            // K ranges per output tile (1: whole K)
    // the last partial round's output tiles split along K (ksplit == 1 only): work units
    // past full_units are (tail tile t, part ks) partials of output tile full_units + t,
    // written densely [BM][BN] to tail_buf + (t * tail_split + ks) * BM * BN
    int full_units, tail_split;
    float *tail_buf;
    int a_rows;            // rows of the A box (BM, or fewer when M is small: the MMA rows past them are unused)
    int tile_start[5];     // prefix sums of tiles per group (ksplit tiles per output tile)
    int n_tiles[4];
    int N[4];
    float *C[4];           // ksplit == 1: the outputs; else partial k of group g at C[g] + k * part_stride
    int64_t ldc[4];
    int64_t part_stride;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait for the completion of the phase with the given parity.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        if ((i & 255u) == 255u) {
            if (*abort) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > g_gemm_wait_ns) {
                *abort = 1;
                atomicOr(&g_gemm_tc_err, 1u);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag: drains copies or MMAs still in
// flight after a give-up, before the CTA frees its TMEM and exits.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return;
        if ((i & 255u) == 255u) {
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kDrainNs) return;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout TMA writes (8-row atoms of 1024 bytes, stride-byte-offset 1024).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)1 << 16;                           // leading-byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                 // stride-byte offset
    d |= (uint64_t)1 << 46;                           // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Work unit -> group, m-tile, n-tile, K-split index and K-split count of its range.
__device__ __forceinline__ void tile_coords(const TcParams &p, int unit, int &g, int &mt, int &nt, int &ks, int &nsplit) {
    int tile = unit;
    nsplit = p.ksplit;
    if (p.tail_split > 1 && unit >= p.full_units) {
        tile = p.full_units + (unit - p.full_units) / p.tail_split;
        nsplit = p.tail_split;
    }
    g = 0;
    while (g + 1 < p.n_groups && tile >= p.tile_start[g + 1]) g++;
    const int local = tile - p.tile_start[g];
    if (nsplit == p.tail_split && p.tail_split > 1) {
        ks = (unit - p.full_units) % p.tail_split;
        nt = local / p.m_tiles;
        mt = local % p.m_tiles;
        return;
    }
    ks = local % p.ksplit;
    const int o = local / p.ksplit;
    nt = o / p.m_tiles;
    mt = o % p.m_tiles;
}

template <int BN, int AR>
__global__ void __launch_bounds__(THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB0,
               const __grid_constant__ CUtensorMap mapB1, const __grid_constant__ CUtensorMap mapB2,
               const __grid_constant__ CUtensorMap mapB3, TcParams p) {
    using G = GT<BN, AR>;
    constexpr int STAGES = G::STAGES, A_BYTES = G::A_BYTES, STAGE_BYTES = G::STAGE_BYTES, TMEM_COLS = G::TMEM_COLS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + G::PAD);
    uint64_t *full = bars, *empty = bars + STAGES, *acc_full = bars + 2 * STAGES, *acc_empty = bars + 2 * STAGES + 2;
    uint64_t *drain = bars + 2 * STAGES + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = p.tail_split > 1 ? p.full_units + (p.tile_start[p.n_groups] - p.full_units) * p.tail_split
                                       : p.tile_start[p.n_groups];
    const int kb_count = (p.K + BK - 1) / BK;
    auto k_range = [&](int ks, int nsplit, int &kb0, int &kb1) {
        const int per = (kb_count + nsplit - 1) / nsplit;
        kb0 = ks * per;
        kb1 = min(kb_count, kb0 + per);
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int a = 0; a < 2; a++) {
            mbar_init(smem_u32(&acc_full[a]), 1);
            mbar_init(smem_u32(&acc_empty[a]), 128);
        }
        mbar_init(smem_u32(drain), 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mapA)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        fence_before();
    }
    __syncthreads();
    fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // TMA producer
            uint32_t it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                int g, mt, nt, ks, nsplit, kb0, kb1;
                tile_coords(p, tile, g, mt, nt, ks, nsplit);
                k_range(ks, nsplit, kb0, kb1);
                const CUtensorMap *mb = g == 0 ? &mapB0 : g == 1 ? &mapB1 : g == 2 ? &mapB2 : &mapB3;
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1, abort)) { ok = false; break; }
                    uint8_t *sa = smem + s * STAGE_BYTES;
                    uint8_t *sb = sa + A_BYTES;
                    const uint32_t bar = smem_u32(&full[s]);
                    mbar_expect_tx(bar, (uint32_t)(p.a_rows * BK * 2 + (STAGE_BYTES - A_BYTES)));
                    tma_load_2d(smem_u32(sa), &mapA, kb * BK, mt * BM, bar);
                    tma_load_2d(smem_u32(sb), mb, kb * BK, nt * BN, bar);
                }
            }
            // after a give-up: the loads still in flight (the last STAGES issued) land before the CTA exits
            if (!ok)
                for (uint32_t u = it > (uint32_t)STAGES ? it - STAGES : 0; u < it; u++)
                    mbar_drain(smem_u32(&full[u % STAGES]), (u / STAGES) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer
            uint32_t it = 0, local = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, local++) {
                const int acc = local & 1;
                const uint32_t aph = (local >> 1) & 1;
                if (!mbar_wait(smem_u32(&acc_empty[acc]), aph ^ 1, abort)) break;
                fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                int g_, mt_, nt_, ks_, ns_, kb0, kb1;
                tile_coords(p, tile, g_, mt_, nt_, ks_, ns_);
                k_range(ks_, ns_, kb0, kb1);
                for (int kb = kb0; kb < kb1; kb++, it++) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&full[s]), ph, abort)) { ok = false; break; }
                    fence_after();
                    const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 16; k++)
                        mma_bf16(d_tmem, sw128_desc(sa + k * 32), sw128_desc(sb + k * 32), G::IDESC,
                                 (kb > kb0 || k > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&empty[s]));
                }
                if (ok) mma_commit(smem_u32(&acc_full[acc]));
            }
            // drain: every MMA issued so far completes (bounded wait, given up or not) before the
            // TMEM is freed: one more commit tracks all of them
            mma_commit(smem_u32(drain));
            mbar_drain(smem_u32(drain), 0);
        }
    } else {
        // epilogue: warps 2..5 -> TMEM lane quarter (warp % 4)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        uint32_t local = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, local++) {
            int g, mt, nt, ks, nsplit;
            tile_coords(p, tile, g, mt, nt, ks, nsplit);
            const int acc = local & 1;
            const uint32_t aph = (local >> 1) & 1;
            if (!mbar_wait(smem_u32(&acc_full[acc]), aph, abort)) break;
            fence_after();
            if (p.tail_split > 1 && tile >= p.full_units) {
                // a tail partial: the whole dense [BM][BN] block, bounds applied by the reduce
                float *trow = p.tail_buf + ((size_t)(tile - p.full_units) * BM + row) * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; c++) {
                    uint32_t r[32];
                    tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
#pragma unroll
                    for (int v = 0; v < 8; v++)
                        *reinterpret_cast<float4 *>(trow + c * 32 + 4 * v) =
                            make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                }
                fence_before();
                mbar_arrive(smem_u32(&acc_empty[acc]));
                continue;
            }
            const int m = mt * BM + row;
            const int n0 = nt * BN;
            float *crow = p.C[g] + (size_t)ks * p.part_stride + (size_t)m * p.ldc[g];
#pragma unroll 1
            for (int c = 0; c < BN / 32; c++) {
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN + c * 32), r);
                const int n = n0 + c * 32;
                if (m < p.M && n < p.N[g]) {
                    if (n + 32 <= p.N[g]) {
#pragma unroll
                        for (int v = 0; v < 8; v++)
                            *reinterpret_cast<float4 *>(crow + n + 4 * v) =
                                make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                            __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                    } else {
                        for (int v = 0; v < 32 && n + v < p.N[g]; v++) crow[n + v] = __uint_as_float(r[v]);
                    }
                }
            }
            fence_before();
            mbar_arrive(smem_u32(&acc_empty[acc]));
        }
    }
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(TMEM_COLS) : "memory");
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool make_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t K, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
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

// The tail tiles' outputs: C = sum over the parts of each tile's dense partials, in part
// order.  One block per (tail tile, group of 8 rows); out-of-range rows and columns are
// dropped.
template <int BN>
__global__ void __launch_bounds__(256) tail_reduce_kernel(const float *__restrict__ tail_buf, TcParams p) {
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x / (BM / 8);
    const int r0 = (blockIdx.x % (BM / 8)) * 8;
    const int tile = p.full_units + t;
    int g = 0;
    while (g + 1 < p.n_groups && tile >= p.tile_start[g + 1]) g++;
    const int local = tile - p.tile_start[g];
    const int nt = local / p.m_tiles, mt = local % p.m_tiles;
    for (int e = threadIdx.x; e < 8 * BN / 4; e += blockDim.x) {
        const int r = r0 + e / (BN / 4), c = (e % (BN / 4)) * 4;
        const int m = mt * BM + r, n = nt * BN + c;
        const float *src = tail_buf + ((size_t)t * p.tail_split * BM + r) * BN + c;
        float4 acc = *reinterpret_cast<const float4 *>(src);
        for (int k = 1; k < p.tail_split; k++) {
            const float4 v = *reinterpret_cast<const float4 *>(src + (size_t)k * BM * BN);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (m >= p.M || n >= p.N[g]) continue;
        float *dst = p.C[g] + (size_t)m * p.ldc[g] + n;
        if (n + 4 <= p.N[g]) {
            *reinterpret_cast<float4 *>(dst) = acc;
        } else {
            const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int v = 0; v < 4 && n + v < p.N[g]; v++) dst[v] = a4[v];
        }
    }
}

// Sum of the split-K partials, in split order: C[m][n] = sum_k part[k][m][n]
// over the whole [M][ldc] block the groups write into.
__global__ void splitk_reduce_kernel(float *__restrict__ C, const float *__restrict__ part, int64_t n4, int64_t stride,
                                     int ksplit) {
    // the dependent kernel may start now (it waits for this grid before reading C); the
    // partials are read only after the GEMM is complete
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 acc = reinterpret_cast<const float4 *>(part)[i];
    for (int k = 1; k < ksplit; k++) {
        const float4 v = reinterpret_cast<const float4 *>(part + (size_t)k * stride)[i];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    reinterpret_cast<float4 *>(C)[i] = acc;
}

template <int BN, int AR>
cudaError_t launch_bn(const GemmArgs &a, cudaStream_t s) {
    using G = GT<BN, AR>;
    if (((uintptr_t)a.A & 15) != 0) return cudaErrorNotSupported;
    TcParams p{};
    p.M = a.M;
    p.K = a.K;
    p.m_tiles = (a.M + BM - 1) / BM;
    p.n_groups = a.n_groups;
    // split K when a partial buffer is given: the split count with the shortest
    // critical path, rounds of work units over the SMs times the time of one unit
    // (its k-blocks plus about two k-blocks of tile setup and partial epilogue);
    // ties go to fewer splits; every split gets at least 4 k-blocks, none is empty
    int ksplit = 1;
    if (a.part && a.c_base) {
        int out_tiles = 0;
        for (int g = 0; g < a.n_groups; g++) out_tiles += p.m_tiles * ((a.g[g].N + BN - 1) / BN);
        const int kb_count = (a.K + BK - 1) / BK;
        const int sms = sm_count();
        constexpr int UNIT_COST = 2;
        long best = (long)((out_tiles + sms - 1) / sms) * (kb_count + UNIT_COST);
        for (int k = 2; k <= a.max_ksplit; k++) {
            const int kb_per = (kb_count + k - 1) / k;
            if (kb_per < 4 || (k - 1) * kb_per >= kb_count) continue;
            // at most three quarters of the SMs: in a decode step the indexer score starts
            // beside this GEMM (its blocks only need SMs the GEMM leaves free)
            if (out_tiles * k > sms * 3 / 4) continue;
            const long cost = (long)((out_tiles * k + sms - 1) / sms) * (kb_per + UNIT_COST);
            if (cost < best) {
                best = cost;
                ksplit = k;
            }
        }
    }
    p.ksplit = ksplit;
    p.part_stride = (int64_t)a.M * a.part_ld;
    p.tail_split = 1;
    CUtensorMap mA, mB[4];
    // small M: a box of the rows present (multiple of 8), not of the whole MMA tile
    p.a_rows = a.M >= BM ? BM : ((a.M + 7) / 8) * 8;
    if (!make_map(&mA, a.A, (uint64_t)a.M, (uint64_t)a.K, (uint32_t)p.a_rows)) return cudaErrorNotSupported;
    int start = 0;
    for (int g = 0; g < 4; g++) {
        const int gi = g < a.n_groups ? g : a.n_groups - 1;
        if (g < a.n_groups) {
            const GemmGroup &G_ = a.g[g];
            if (((uintptr_t)G_.B & 15) != 0 || (G_.ldc % 4) != 0 || ((uintptr_t)G_.C & 15) != 0) return cudaErrorNotSupported;
            if (!make_map(&mB[g], G_.B, (uint64_t)G_.N, (uint64_t)a.K, BN)) return cudaErrorNotSupported;
            p.N[g] = G_.N;
            p.C[g] = ksplit > 1 ? a.part + (G_.C - a.c_base) : G_.C;
            p.ldc[g] = G_.ldc;
            p.n_tiles[g] = (G_.N + BN - 1) / BN;
            p.tile_start[g] = start;
            start += p.n_tiles[g] * p.m_tiles * ksplit;
        } else {
            mB[g] = mB[gi];
        }
    }
    p.tile_start[a.n_groups] = start;
    p.full_units = start;
    // a last round that fills at most half the SMs: its tiles split along K over the SMs
    // (every part at least 4 k-blocks, none empty), partials summed by tail_reduce_kernel
    if (ksplit == 1 && a.tail_buf && BN == 256) {
        const int sms = sm_count();
        const int rounds = (start + sms - 1) / sms;
        const int tail = start - (rounds - 1) * sms;
        const int kb_count = (a.K + BK - 1) / BK;
        if (rounds >= 2 && 2 * tail <= sms) {
            int split = sms / tail;
            if (split > kb_count / 4) split = kb_count / 4;
            while (split >= 2 && (split - 1) * ((kb_count + split - 1) / split) >= kb_count) split--;
            if (split >= 2) {
                p.full_units = start - tail;
                p.tail_split = split;
                p.tail_buf = a.tail_buf;
            }
        }
    }
    if (p.a_rows > AR) return cudaErrorInvalidValue;
    cudaError_t e = ensure_dyn_smem(gemm_tc_kernel<BN, AR>, G::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int units = p.tail_split > 1 ? p.full_units + (start - p.full_units) * p.tail_split : start;
    const int grid = units < sm_count() ? units : sm_count();
    e = launch_pdl(gemm_tc_kernel<BN, AR>, dim3(grid), dim3(THREADS), G::SMEM_BYTES, s, mA, mB[0], mB[1], mB[2], mB[3], p);
    if (e == cudaSuccess && p.tail_split > 1)
        return launch_pdl(tail_reduce_kernel<BN>, dim3((unsigned)((start - p.full_units) * (BM / 8))), dim3(256), 0, s,
                          (const float *)p.tail_buf, p);
    if (e != cudaSuccess || ksplit == 1) return e;
    const int64_t n4 = (int64_t)a.M * a.part_ld / 4;
    return launch_pdl(splitk_reduce_kernel, dim3((unsigned)((n4 + 255) / 256)), dim3(256), 0, s, a.c_base,
                      (const float *)a.part, n4, p.part_stride, ksplit);
}

}  // namespace

size_t gemm_tail_floats() { return (size_t)sm_count() * BM * 256; }

cudaError_t launch_gemm_tc(const GemmArgs &a, cudaStream_t s) {
    if (a.dtype != DS4C_BF16 || a.M < 1 || a.K % 8 != 0 || a.n_groups < 1 || a.n_groups > 4)
        return cudaErrorNotSupported;
    if (((uintptr_t)a.A & 15) != 0) return cudaErrorNotSupported;
    // decode-sized M: narrow tiles, so the weight traffic spreads over many SMs
    // at most 32 rows: wide tiles (fewer re-reads of the activations per weight
    // byte) over thin stages, split along K to cover the SMs
    if (a.M <= 32) return launch_bn<128, 32>(a, s);
    return a.M <= 256 ? launch_bn<32, BM>(a, s) : launch_bn<256, BM>(a, s);
}

cudaError_t gemm_tc_set_wait_ns(unsigned long long ns) { return cudaMemcpyToSymbol(g_gemm_wait_ns, &ns, sizeof ns); }

unsigned int gemm_tc_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_tc_err, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_gemm_tc_err, &z, sizeof z);
    return v;
}

}  // namespace ds4c
