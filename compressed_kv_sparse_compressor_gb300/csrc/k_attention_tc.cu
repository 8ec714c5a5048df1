// Sparse sliding-window attention on the 5th-generation tensor cores (K6),
// "Metal グラフと圧縮 KV の実装を読む" §7: per query position t and head h one
// softmax over the raw window rows and the compressed rows the layer selects,
// K = V = the stored row, all heads sharing it.
//
// Formulation (one query token at a time, all H heads together):
//   S^T[r][h | H+h] = sum_d X[r][d] [Q_hi | Q_lo][h][d]   M = 128 rows, N = 2H, K = D
//   O^T[d][h] += sum_r X[r][d] P[r][h]                   M = 128 d (D/128 blocks), N = H, K = rows
//   L[h] += sum_r P[r][h]                                (the softmax denominator, on the CUDA cores)
// Rows sit on TMEM lanes, heads on TMEM columns.  Accuracy: every operand is
// split into bf16 hi + lo (x = hi + lo to 2^-17) and each product takes the
// three parts hi*hi + hi*lo + lo*hi, fp32 accumulation in tensor memory; this
// keeps the result within fp32-accumulation tolerance of the exact attention.
// The S product multiplies X by Q_hi and Q_lo in one N = 2H MMA (the two halves
// land side by side in TMEM and the softmax adds them), so the X operand is
// read from shared memory once for both.
//
// Data: row tiles arrive from bf16 hi/lo mirrors: raw rows by TMA from a
// position-ordered mirror the call builds in the workspace (one 128-row box per
// query), compressed rows from the comp_split mirror the compressor maintains,
// gathered by the row list (top-k on ratio-4 layers, every visible row on
// ratio-128 layers) with 16-byte cp.async by the two producer warps into the
// same 128-byte-swizzled layout, eight lanes copying one row's 128 bytes so
// that an instruction reads four whole lines (on the six 32 KB slots below
// this beat lane pairs sharing 32-byte sectors, sixteen rows per instruction,
// by 9 %; on an earlier ring of 16 KB slots it had been the slower one).  A
// tile is streamed twice through a ring of six 32 KB slots: by 64-wide
// d-chunks for S (each slot with the query chunk it meets), by 128-wide
// d-blocks for O (the same bytes form the K-major A operand of the first
// product and the MN-major A operand of the second).  Compressed rows
// went through the E4M3 round trip on their first head_dim - n_rot dims, so
// those values are exact in bf16 and their lo half is zero: the lo loads and
// the lo MMAs of those dims are skipped.
//
// Softmax: online with a lazy reference maximum: a tile only moves the
// reference (and rescales O and L in tensor memory) when a logit exceeds it by
// more than 2^8, so p <= 256 and the final O/L is exact for any reference.
//
// Warp roles (384 threads in three warpgroups, persistent over query tokens):
//   warps 0, 2  row lists and producers    warp 1  MMA issuer, TMEM owner   (warp 3 idle)
//   warps 4-7   softmax and P (thread = TMEM lane = tile row)
//   warps 8-11  Q loader and epilogue (thread = TMEM lane = d within a block): the next
//               query's Q is loaded and split as soon as the current query's last S has
//               been computed, and the output is read out of tensor memory and stored
//               while the softmax and the MMAs carry on with the next query; only the
//               first O product of the next query waits, block by block, for the read.
// The warpgroups resize their register files at entry (setmaxnreg) so that the softmax
// holds its 64 logits and a block of O without spilling.
// Every mbarrier wait is bounded; a wait that gives up raises the device error
// word and the CTA winds down.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ds4c_internal.cuh"

namespace ds4c {

__device__ unsigned int g_attn_tc_err;
__device__ unsigned long long g_attn_wait_ns = kWaitNsDefault;

namespace {

constexpr int ROWS = 128;
constexpr int SLOT = 8192;            // [64 rows][64 d] bf16
constexpr int PAIR = 2 * SLOT;
constexpr int USLOT = 2 * PAIR;      // one ring slot
constexpr int RING = 6;
// three warpgroups: {producer, MMA, two idle warps}, the softmax, the Q loader / epilogue
constexpr int THREADS = 384;
// registers per thread after the reallocation at entry (setmaxnreg): the first warpgroup gives
// up registers, the softmax warpgroup takes them, the third keeps its launch allocation.  The
// launch allocation must be at least (REG_LOW + REG_SOFT) / 2 for the two to fit (host-checked).
constexpr int REG_LOW = 128;
constexpr int REG_SOFT = 240;
constexpr int REG_AUX = 136;
constexpr int MAX_LIST = 512;
constexpr float TAU = 8.0f;           // log2 units

template <int H, int D>
struct L {
    static constexpr int DC = D / 64;
    static constexpr int DB = D / 128;
    static constexpr int PB = ROWS * H * 2;            // bytes of P hi (or lo)
    // the ring: 16 KB units of gathered rows, raw-row boxes and query chunks (a query
    // chunk [2H][64] bf16 holds Q_hi of 64 d in rows 0 .. H-1 and Q_lo in rows H .. 2H-1)
    static constexpr int OFF_X = 0;
    static constexpr int OFF_PHI = OFF_X + RING * USLOT;
    static constexpr int OFF_PLO = OFF_PHI + PB;
    static constexpr int OFF_LIST = OFF_PLO + PB;
    // per head: the tile maximum as an order-preserving key, then (same word)
    // the rescale factor of the new reference
    static constexpr int OFF_TMAX = OFF_LIST + 4 * MAX_LIST;
    static constexpr int OFF_MREF = OFF_TMAX + 4 * H;
    static constexpr int OFF_FLAG = OFF_MREF + 4 * H;
    // per head: the softmax denominator of the item the epilogue writes
    static constexpr int OFF_LFIN = OFF_FLAG + 8;
    static constexpr int OFF_BAR = OFF_LFIN + 4 * H;
    static constexpr int N_BAR = 2 * RING + 16;
    static_assert(2 * H * 64 * 2 == PAIR, "a query chunk fills half a ring slot");
    // the dynamic shared memory starts 1024-byte aligned (checked at entry), as
    // the 128-byte swizzle atoms of Q, the ring and P need
    static constexpr int SMEM = OFF_BAR + 8 * N_BAR + 16;
    // TMEM columns
    static constexpr int T_S = 0;                      // two S^T buffers of 2H columns (Q_hi part | Q_lo part)
    static constexpr int T_O = 4 * H;                  // DB blocks of H columns
    static constexpr int T_COLS = 512;
    static_assert(T_O + DB * H <= T_COLS, "tensor memory");
    static_assert(SMEM <= 232448, "shared memory");
    static_assert(DB <= 4, "one output-free barrier per pair of d-blocks");
};

// barrier indices
enum { B_FULL = 0, B_EMPTY = RING, B_QREADY0 = 2 * RING, B_QREADY1, B_SFULL0, B_SFULL1, B_SFREE0, B_SFREE1, B_PFULL,
       B_PVDONE, B_OFREE0, B_OFREE1, B_SOFT, B_DRAIN, B_QFREE0, B_QFREE1, B_LREADY, B_PBAR, B_COUNT };
// barriers indexed as X0 + parity must be adjacent
static_assert(B_QREADY1 == B_QREADY0 + 1 && B_SFULL1 == B_SFULL0 + 1 && B_SFREE1 == B_SFREE0 + 1 &&
                  B_OFREE1 == B_OFREE0 + 1 && B_QFREE1 == B_QFREE0 + 1,
              "barrier pairs indexed by a parity are adjacent");
static_assert(B_COUNT == 2 * RING + 16, "the layout's barrier count");

struct TcAttnParams {
    float *out;                      // this launch's first head of out[n_q][..][D], o_ld floats per query
    const float *q;                  // this launch's first head of q[n_q][..][D], q_ld floats per query
    int64_t q_ld, o_ld;
    int nh;                          // heads of this launch (<= H: the kernel runs H, the rest padded)
    uint16_t *qsplit;                // per CTA two buffers [D/64][2H][64] bf16 of split queries, or (qpre)
                                     // every query's [D/64][2H][64], split before the launch
    int qpre;
    const int32_t *topk;
    const uint16_t *comp_split;      // [rows][2][D]
    int n_q, n_seq, n_tok, k, ratio, comp_cap;
    int swa;                         // raw window (ring rows), at most 128: the raw tile's valid rows
    int nope_chunks, nope_blocks;    // 64-wide chunks / 128-wide blocks inside the FP8 dims
    int parts;                       // work items per query (1: whole query; >1: split rows, partial outputs)
    float *part_o;                   // [n_q * parts][nh][D] unnormalised partial outputs
    float *part_ml;                  // [n_q * parts][2][nh] reference max (log2) and denominator
    float scale_log2;
    uint64_t pos0;
    DecodePos dp;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// the bytes a phase still waits for, without an arrival
__device__ __forceinline__ void mbar_expect_tx_only(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Each poll may suspend the thread for up to 1 us (woken when the phase completes), so a waiting
// warp does not keep issuing beside the MMA warp; the time is checked every 16 polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(1000u)
            : "memory");
        if (ok) return true;
        if ((i & 15u) == 15u) {
            if (*abort) return false;
            const uint64_t now = globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > g_attn_wait_ns) {
                *abort = 1;
                atomicOr(&g_attn_tc_err, 1u);
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

__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05) with the start address left zero: leading /
// stride byte offsets, version 1, layout (2 = 128-byte swizzle).  Adding (address >> 4)
// fills in the start (shared-memory addresses are below 256 KB, so the sum stays inside
// the 14-bit field).
__host__ __device__ constexpr uint64_t desc_template(uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) |
           ((uint64_t)layout << 61);
}

// Instruction descriptor, kind::f16 with bf16 operands and f32 accumulation.
__host__ __device__ constexpr uint32_t idesc(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// The same two issued by a converged warp: every lane computes the (warp-uniform) operands and
// only the lane with `leader` set issues, so one thread issues every MMA and every commit.
__device__ __forceinline__ void mma_w(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc,
                                      uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 e, %5, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(acc), "r"(leader)
        : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint32_t bar, uint32_t leader) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "setp.ne.b32 e, %1, 0;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
        "r"(leader)
        : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// the barrier counts one arrival when this thread's earlier cp.async copies land
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

#define TMEM_LD16(taddr, r, o)                                                                                    \
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, " \
                 "%13, %14, %15}, [%16];"                                                                        \
                 : "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]),   \
                   "=r"(r[o + 6]), "=r"(r[o + 7]), "=r"(r[o + 8]), "=r"(r[o + 9]), "=r"(r[o + 10]), "=r"(r[o + 11]), \
                   "=r"(r[o + 12]), "=r"(r[o + 13]), "=r"(r[o + 14]), "=r"(r[o + 15])                              \
                 : "r"(taddr))
#define TMEM_ST16(taddr, r, o)                                                                                     \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, " \
                 "%13, %14, %15, %16};" ::"r"(taddr),                                                             \
                 "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), "r"(r[o + 4]), "r"(r[o + 5]),           \
                 "r"(r[o + 6]), "r"(r[o + 7]), "r"(r[o + 8]), "r"(r[o + 9]), "r"(r[o + 10]), "r"(r[o + 11]),        \
                 "r"(r[o + 12]), "r"(r[o + 13]), "r"(r[o + 14]), "r"(r[o + 15])                                   \
                 : "memory")

// Load H consecutive fp32 columns of this thread's TMEM lane.
template <int H>
__device__ __forceinline__ void tmem_load(uint32_t taddr, float (&v)[H]) {
    uint32_t r[H];
#pragma unroll
    for (int c = 0; c < H; c += 16) TMEM_LD16(taddr + c, r, c);
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int c = 0; c < H; c++) v[c] = __uint_as_float(r[c]);
}
template <int H>
__device__ __forceinline__ void tmem_store(uint32_t taddr, const float (&v)[H]) {
    uint32_t r[H];
#pragma unroll
    for (int c = 0; c < H; c++) r[c] = __float_as_uint(v[c]);
#pragma unroll
    for (int c = 0; c < H; c += 16) TMEM_ST16(taddr + c, r, c);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// S of this thread's row: the Q_hi and the Q_lo halves of the N = 2H product
// added, 16 columns at a time (keeps the register footprint at H + 32).
template <int H>
__device__ __forceinline__ void tmem_load_s(uint32_t taddr, float (&v)[H]) {
#pragma unroll
    for (int c = 0; c < H; c += 16) {
        uint32_t a[16], b[16];
        TMEM_LD16(taddr + c, a, 0);
        TMEM_LD16(taddr + H + c, b, 0);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int j = 0; j < 16; j++) v[c + j] = __uint_as_float(a[j]) + __uint_as_float(b[j]);
    }
}

// Warp reduction over the 32 rows of a warp of 64 per-head values, by a
// transposing butterfly: at offset o each lane keeps the half of its heads
// selected by lane bit o and takes the partner's values for it, so that after
// the five steps lane l holds heads 2l (r0) and 2l + 1 (r1).  v is only read.
template <bool MAX>
__device__ __forceinline__ void warp_heads_reduce(const float (&v)[64], float &r0, float &r1) {
    const int lane = threadIdx.x & 31;
    float m[32];
    {
        const bool up = (lane & 16) != 0;
#pragma unroll
        for (int k = 0; k < 32; k++) {
            const float send = up ? v[k] : v[k + 32];
            const float keep = up ? v[k + 32] : v[k];
            const float o = __shfl_xor_sync(0xffffffffu, send, 16);
            m[k] = MAX ? fmaxf(keep, o) : keep + o;
        }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < 2 * o; k++) {
            const float send = up ? m[k] : m[k + 2 * o];
            const float keep = up ? m[k + 2 * o] : m[k];
            const float x = __shfl_xor_sync(0xffffffffu, send, o);
            m[k] = MAX ? fmaxf(keep, x) : keep + x;
        }
    }
    r0 = m[0];
    r1 = m[1];
}

// order-preserving u32 image of a float (for atomicMax) and back
__device__ __forceinline__ uint32_t max_key(float x) {
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_max(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo) {
    hi = __bfloat162float(__float2bfloat16_rn(x));
    lo = x - hi;
}

// Per-token geometry shared by all roles.
struct Tok {
    int n;             // query index
    int seq;
    uint64_t t;        // position
    int raw_row0;      // raw mirror row of tile 0, row 0
    int raw_lo, raw_hi;  // valid row range of tile 0
    int n_comp;
    int n_tiles;
};

__device__ __forceinline__ Tok token_geom(const TcAttnParams &p, int n) {
    Tok k;
    k.n = n;
    if (p.n_seq == 1) {
        k.seq = 0;
        k.t = p.pos0 + (uint64_t)n;
        k.raw_row0 = n + 1;                               // mirror row u <-> position pos0 - 128 + u
        // the window's positions t - swa + 1 .. t (from 0 on) are the tile's last rows
        k.raw_lo = ROWS - 1 - (int)(k.t < (uint64_t)(p.swa - 1) ? k.t : (uint64_t)(p.swa - 1));
        k.raw_hi = ROWS - 1;
    } else {
        k.seq = n;
        k.t = p.dp.pos[n];
        k.raw_row0 = n * ROWS;                            // mirror rows = the sequence's swa ring slots, then zeros
        k.raw_lo = 0;
        k.raw_hi = k.t < (uint64_t)(p.swa - 1) ? (int)k.t : p.swa - 1;   // slot s holds position s while t < swa
    }
    return k;
}

// Number of compressed rows a query attends (ratio 4: the top-k list read the
// way the attention loop of [P2] §7 reads it -- entries < 0 skipped, the first
// entry >= visible ends the list; ratio 128: every visible row).  The whole
// warp calls this; each lane loads 16 consecutive entries at once, so a 512-
// entry list costs one memory latency.  The list (row indices into the comp
// mirror) is written to `list` when non-null.
__device__ __forceinline__ int comp_rows(const TcAttnParams &p, const Tok &k, int *list) {
    const int lane = threadIdx.x & 31;
    if (p.ratio == 128) {
        const uint64_t v = (k.t + 1) / 128;
        return v < (uint64_t)p.comp_cap ? (int)v : p.comp_cap;
    }
    if (p.ratio != 4) return 0;
    const uint64_t visible = (k.t + 1) / 4;
    const int32_t *tk = p.topk + (size_t)k.n * p.k;
    int cnt = 0;
    for (int base = 0; base < p.k; base += 512) {
        int32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const int i = base + lane * 16 + j;
            v[j] = (i < p.k) ? __ldg(tk + i) : -1;
        }
        int first_stop = 16, local = 0;
#pragma unroll
        for (int j = 0; j < 16; j++) {
            const bool stop = v[j] >= 0 && (uint64_t)v[j] >= visible;
            if (stop && first_stop == 16) first_stop = j;
            if (v[j] >= 0 && first_stop == 16) local++;
        }
        const unsigned stop_m = __ballot_sync(0xffffffffu, first_stop < 16);
        const int f = stop_m ? __ffs(stop_m) - 1 : 32;     // first lane holding a stop
        const int contrib = lane < f ? local : (lane == f ? local : 0);
        // exclusive prefix of the contributions
        int incl = contrib;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (list && contrib > 0) {
            int w = cnt + incl - contrib;
#pragma unroll
            for (int j = 0; j < 16; j++)
                if (j < first_stop && v[j] >= 0) list[w++] = k.seq * p.comp_cap + v[j];
        }
        cnt += __shfl_sync(0xffffffffu, incl, 31);
        if (stop_m) break;
    }
    return cnt;
}

// Work item `it` = (query it / parts, part it % parts); the part covers tiles
// [tb, te) of its query (empty when tb >= te).
struct Item { int n, tb, te; };
__device__ __forceinline__ Item item_tiles(const TcAttnParams &p, int it, int n_tiles) {
    Item r;
    r.n = it / p.parts;
    const int part = it % p.parts;
    if (p.parts == 1) {
        r.tb = 0;
        r.te = n_tiles;
        return r;
    }
    // split rows: the raw tile alone (its lo halves make it the longest), the compressed
    // tiles spread evenly over the other parts
    if (part == 0) {
        r.tb = 0;
        r.te = 1;
        return r;
    }
    const int w = (n_tiles - 1 + p.parts - 2) / (p.parts - 1);
    r.tb = 1 + (part - 1) * w;
    r.te = min(r.tb + w, n_tiles);
    return r;
}

// Next work item of this CTA at or after `it` that has rows (n_items when
// none).  The whole warp calls this.
__device__ __forceinline__ int next_item(const TcAttnParams &p, int it, int n_items) {
    for (; it < n_items; it += gridDim.x) {
        const Tok kk = token_geom(p, it / p.parts);
        const int ncc = comp_rows(p, kk, nullptr);
        const Item ii = item_tiles(p, it, 1 + (ncc + ROWS - 1) / ROWS);
        if (ii.tb < ii.te) return it;
    }
    return n_items;
}

template <int H, int D>
__global__ void __launch_bounds__(THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap rawHi, const __grid_constant__ CUtensorMap rawLo,
               const __grid_constant__ CUtensorMap qsMap, const TcAttnParams p) {
    using Lay = L<H, D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if ((smem_u32(smem_raw) & 1023u) != 0) {            // the layout has no room to realign
        pdl_wait();                                      // keep the launch chain ordered
        if (threadIdx.x == 0) atomicOr(&g_attn_tc_err, 4u);
        return;
    }
    uint8_t *sm = smem_raw;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + Lay::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Lay::N_BAR);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *list = reinterpret_cast<int *>(sm + Lay::OFF_LIST);
    uint32_t *tmax = reinterpret_cast<uint32_t *>(sm + Lay::OFF_TMAX);
    float *alpha_s = reinterpret_cast<float *>(sm + Lay::OFF_TMAX);
    float *mref_s = reinterpret_cast<float *>(sm + Lay::OFF_MREF);
    volatile uint8_t *flags = reinterpret_cast<volatile uint8_t *>(sm + Lay::OFF_FLAG);
    float *lfin = reinterpret_cast<float *>(sm + Lay::OFF_LFIN);
    auto bar = [&](int i) { return smem_u32(&bars[i]); };

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < RING; i++) {
            mbar_init(bar(B_FULL + i), 64);        // one arrival per lane of the two producer warps
            mbar_init(bar(B_EMPTY + i), 1);
        }
        mbar_init(bar(B_QREADY0), 128);
        mbar_init(bar(B_QREADY1), 128);
        mbar_init(bar(B_SFULL0), 1);
        mbar_init(bar(B_SFULL1), 1);
        mbar_init(bar(B_SFREE0), 128);
        mbar_init(bar(B_SFREE1), 128);
        mbar_init(bar(B_PFULL), 128);
        mbar_init(bar(B_PVDONE), 1);
        for (int j = 0; j < 2; j++) mbar_init(bar(B_OFREE0 + j), 128);
        mbar_init(bar(B_SOFT), 128);
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_QFREE0), 1);
        mbar_init(bar(B_QFREE1), 1);
        mbar_init(bar(B_LREADY), 128);
        mbar_init(bar(B_PBAR), 64);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(Lay::T_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        fence_before();
    }
    fence_proxy_async();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    pdl_launch_dependents();

    // Each warpgroup first resizes its register allocation (setmaxnreg, one instruction for its
    // four warps, which the code of the role then follows); the host checked that the three
    // shares fit the launch allocation.
    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_LOW));
    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producer pair
        // warps 0 and 2 share every unit: each copies the 16-row blocks of its parity, and
        // both count on the unit's barrier; the row list is written by warp 0 between two
        // barriers of the pair (the previous list read by both, the new one complete)
        const int pw = warp >> 1;
        uint32_t unit = 0, pphase = 0, tok = 0;
        bool ok = true;
        auto pair_bar = [&]() -> bool {
            mbar_arrive(bar(B_PBAR));
            const bool r_ = mbar_wait(bar(B_PBAR), pphase, abort);
            pphase ^= 1;
            return r_;
        };
        const int n_items = p.n_q * p.parts;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Tok k = token_geom(p, it / p.parts);
            if (!pair_bar()) { ok = false; break; }
            const int nc = comp_rows(p, k, (p.ratio == 4 && pw == 0) ? list : nullptr);
            __syncwarp();
            if (!pair_bar()) { ok = false; break; }
            const Item itm = item_tiles(p, it, 1 + (nc + ROWS - 1) / ROWS);
            if (itm.tb >= itm.te) continue;
            // this item's split query (buffer tok & 1 of this CTA) has been written
            const int qbuf = tok & 1;
            if (pw == 0) {
                int okq = 1;
                if (lane == 0) okq = mbar_wait(bar(B_QREADY0 + qbuf), (tok >> 1) & 1, abort) ? 1 : 0;
                if (__shfl_sync(0xffffffffu, okq, 0) == 0) { ok = false; break; }
            }
            tok++;
            const int qrow0 = (p.qpre ? it / p.parts : blockIdx.x * 2 + qbuf) * Lay::DC * 2 * H;
            const int dummy = k.seq * p.comp_cap;
            auto row_of = [&](int tile, int r) -> int {   // comp mirror row of tile >= 1, row r
                const int i = (tile - 1) * ROWS + r;
                if (i >= nc) return dummy;
                return p.ratio == 4 ? list[i] : dummy + i;
            };
            // this lane's rows 8 i + 4 pw + lane / 8 (i = 0 .. 15): every slot of a compressed tile
            // copies from them, so their mirror rows are looked up once per tile
            int rix[16];
            int rp_tile = -1;
            auto tile_rows = [&](int tile) {
                if (tile == rp_tile) return;
                rp_tile = tile;
#pragma unroll
                for (int i = 0; i < 16; i++) rix[i] = row_of(tile, 8 * i + 4 * pw + (lane >> 3));
            };
            // this warp's half of 16 KB of gathered compressed rows at dst, in the 128-byte swizzle
            // layout: (pv = false) rows 0 .. 127 of the 64-d chunk at element offset off; (pv =
            // true) rows 64 hh .. 64 hh + 63 of the 128-d block at off, as two [64][64] halves
            // SLOT apart.  Eight lanes copy one row's 128 bytes, so an instruction reads four
            // whole lines.
            auto gather16 = [&](uint32_t dst, int tile, bool pv, int off, int hh) {
                tile_rows(tile);
                const int u = lane & 7;                      // 16-byte unit of the row's 128 bytes
                const int sw = (4 * pw + (lane >> 3)) & 7;   // row & 7 of every row this lane copies
                if (!pv) {
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        const int r = 8 * i + 4 * pw + (lane >> 3);
                        const uint16_t *src = p.comp_split + (size_t)rix[i] * 2 * D + off + 8 * u;
                        cp_async16(dst + r * 128 + ((u ^ sw) << 4), src);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const int rr = 8 * i + 4 * pw + (lane >> 3);
                        const int ri = hh ? rix[8 + i] : rix[i];
                        const uint16_t *src = p.comp_split + (size_t)ri * 2 * D + off + 8 * u;
#pragma unroll
                        for (int half = 0; half < 2; half++)
                            cp_async16(dst + half * SLOT + rr * 128 + ((u ^ sw) << 4), src + 64 * half);
                    }
                }
            };
            // the next 32 KB slot of the ring, once the MMAs of its previous contents are done
            auto open_slot = [&](uint32_t &dst, uint32_t &fb) -> bool {
                const int s_ = unit % RING;
                const uint32_t ph = (unit / RING) & 1;
                unit++;
                int okw = 1;
                if (lane == 0) okw = mbar_wait(bar(B_EMPTY + s_), ph ^ 1, abort) ? 1 : 0;
                if (__shfl_sync(0xffffffffu, okw, 0) == 0) {
                    unit--;                                  // nothing was issued for this slot
                    return false;
                }
                dst = smem_u32(sm + Lay::OFF_X + s_ * USLOT);
                fb = bar(B_FULL + s_);
                return true;
            };
            // A slot's barrier takes one arrival per lane of the pair (a lane that gathered arrives
            // when its copies land) plus the bytes of the slot's TMA boxes, which lane 0 of warp 0
            // announces before issuing them.
            const bool lead = pw == 0 && lane == 0;
            // S operands of chunk c: [query chunk c | hi of the rows' chunk c]
            auto slot_qk = [&](int tile, int c) -> bool {
                uint32_t dst, fb;
                if (!open_slot(dst, fb)) return false;
                if (tile == 0) {
                    if (lead) {
                        mbar_expect_tx_only(fb, USLOT);
                        tma_box(dst, &qsMap, 0, qrow0 + c * 2 * H, fb);
                        tma_box(dst + PAIR, &rawHi, 64 * c, k.raw_row0, fb);
                        tma_box(dst + PAIR + SLOT, &rawHi, 64 * c, k.raw_row0 + 64, fb);
                    }
                    mbar_arrive(fb);
                } else {
                    if (lead) {
                        mbar_expect_tx_only(fb, PAIR);
                        tma_box(dst, &qsMap, 0, qrow0 + c * 2 * H, fb);
                    }
                    gather16(dst + PAIR, tile, false, 64 * c, 0);
                    cp_async_arrive(fb);
                }
                return true;
            };
            // lo of the rows' chunks c0 and c1 (c1 < 0: none): [lo c0 | lo c1]
            auto slot_qk_lo = [&](int tile, int c0, int c1) -> bool {
                uint32_t dst, fb;
                if (!open_slot(dst, fb)) return false;
                if (tile == 0) {
                    if (lead) {
                        mbar_expect_tx_only(fb, c1 >= 0 ? USLOT : PAIR);
                        tma_box(dst, &rawLo, 64 * c0, k.raw_row0, fb);
                        tma_box(dst + SLOT, &rawLo, 64 * c0, k.raw_row0 + 64, fb);
                        if (c1 >= 0) {
                            tma_box(dst + PAIR, &rawLo, 64 * c1, k.raw_row0, fb);
                            tma_box(dst + PAIR + SLOT, &rawLo, 64 * c1, k.raw_row0 + 64, fb);
                        }
                    }
                    mbar_arrive(fb);
                } else {
                    gather16(dst, tile, false, D + 64 * c0, 0);
                    if (c1 >= 0) gather16(dst + PAIR, tile, false, D + 64 * c1, 0);
                    cp_async_arrive(fb);
                }
                return true;
            };
            // O operands of d-block j, hi (lo = 0) or lo (lo = 1): [rows 0 .. 63 | rows 64 .. 127]
            auto slot_pv = [&](int tile, int j, int lo) -> bool {
                uint32_t dst, fb;
                if (!open_slot(dst, fb)) return false;
                if (tile == 0) {
                    if (lead) {
                        const CUtensorMap *m = lo ? &rawLo : &rawHi;
                        mbar_expect_tx_only(fb, USLOT);
                        for (int hh = 0; hh < 2; hh++) {
                            tma_box(dst + hh * PAIR, m, 128 * j, k.raw_row0 + 64 * hh, fb);
                            tma_box(dst + hh * PAIR + SLOT, m, 128 * j + 64, k.raw_row0 + 64 * hh, fb);
                        }
                    }
                    mbar_arrive(fb);
                } else {
                    gather16(dst, tile, true, lo * D + 128 * j, 0);
                    gather16(dst + PAIR, tile, true, lo * D + 128 * j, 1);
                    cp_async_arrive(fb);
                }
                return true;
            };
            // the S slots of a tile: every chunk's, each lo chunk pair's (or a last single one's)
            // right after the pair's second chunk
            auto issue_qk = [&](int tile) -> bool {
                const int c0 = tile == 0 ? 0 : p.nope_chunks;     // the first chunk with a lo half
                for (int c = 0; c < Lay::DC; c++) {
                    if (!slot_qk(tile, c)) return false;
                    if (c >= c0) {
                        if ((c - c0) & 1) {
                            if (!slot_qk_lo(tile, c - 1, c)) return false;
                        } else if (c == Lay::DC - 1) {
                            if (!slot_qk_lo(tile, c, -1)) return false;
                        }
                    }
                }
                return true;
            };
            auto issue_pv = [&](int tile) -> bool {
                for (int j = 0; j < Lay::DB; j++) {
                    if (!slot_pv(tile, j, 0)) return false;
                    if ((tile == 0 || j >= p.nope_blocks) && !slot_pv(tile, j, 1)) return false;
                }
                return true;
            };
            bool good = issue_qk(itm.tb);
            for (int i = itm.tb; i < itm.te && good; i++) {
                if (i + 1 < itm.te) good = issue_qk(i + 1);
                if (good) good = issue_pv(i);
            }
            ok = good;
        }
        if (!ok) {
            // after a give-up: this lane's row copies complete, and every unit issued to the ring
            // (the last RING at most are still open) has landed before the CTA exits
            asm volatile("cp.async.wait_all;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                for (uint32_t u = unit > (uint32_t)RING ? unit - RING : 0; u < unit; u++)
                    mbar_drain(bar(B_FULL + u % RING), (u / RING) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t ID_QK = idesc(128, H, 0, 0);
        constexpr uint32_t ID_QK2 = idesc(128, 2 * H, 0, 0);
        constexpr uint32_t ID_PV = idesc(128, H, 1, 1);
        constexpr uint64_t DK = desc_template(16, 1024, 2);      // S operands
        constexpr uint64_t DA = desc_template(SLOT, 1024, 2);    // X^T of the O product
        constexpr uint64_t DP = desc_template(8192, 1024, 2);    // P^T
        const uint32_t phi = smem_u32(sm + Lay::OFF_PHI), plo = smem_u32(sm + Lay::OFF_PLO);
        uint32_t unit = 0, g = 0, tok = 0;
        bool ok = true;
        // The whole warp runs the issue loop (its operands stay warp-uniform); lane 0 issues.
        const uint32_t leader = lane == 0;
        auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(b, parity, abort)) != 0;
        };
        // slot u of the ring: wait until loaded / hand back once its MMAs finish
        auto wait_slot = [&](uint32_t u, uint32_t &base) -> bool {
            base = smem_u32(sm + Lay::OFF_X + (u % RING) * USLOT);
            return wait_all(bar(B_FULL + u % RING), (u / RING) & 1);
        };
        auto free_slot = [&](uint32_t u) { mma_commit_w(bar(B_EMPTY + u % RING), leader); };
        // S of global tile gt; `last`: the item's last tile, after which its query chunks are
        // no longer read.  The slots of a lo chunk pair's query chunks stay held until the
        // pair's lo product has been issued.
        auto do_qk = [&](uint32_t gt, int tile, bool last) -> bool {
            const int sb = gt & 1;
            if (gt >= 2 && !wait_all(bar(B_SFREE0 + sb), ((gt >> 1) - 1) & 1)) return false;
            fence_after();
            const uint32_t d_t = tmem + Lay::T_S + sb * 2 * H;
            const int c0 = tile == 0 ? 0 : p.nope_chunks;
            uint32_t hu0 = 0, hb0 = 0, hu1 = 0, hb1 = 0;   // held slots (index, address)
            int nheld = 0;
            for (int c = 0; c < Lay::DC; c++) {
                uint32_t b;
                if (!wait_slot(unit, b)) return false;
                fence_proxy_async();
                fence_after();
                // K-major operands, 32 bytes (2 descriptor units) per K step of 16: the rows' hi
                // against [Q_hi; Q_lo] (rows 0 .. 2H-1 of the query chunk)
                const uint64_t q0 = DK + (b >> 4), x0 = DK + ((b + PAIR) >> 4);
#pragma unroll
                for (int kk = 0; kk < 4; kk++)
                    mma_w(d_t, x0 + 2 * kk, q0 + 2 * kk, ID_QK2, (c > 0 || kk > 0) ? 1u : 0u, leader);
                const uint32_t mu = unit++;
                if (c < c0) {
                    free_slot(mu);
                    continue;
                }
                if (nheld == 0) { hu0 = mu; hb0 = b; } else { hu1 = mu; hb1 = b; }
                nheld++;
                if (((c - c0) & 1) || c == Lay::DC - 1) {
                    // the rows' lo of the held chunks against Q_hi
                    uint32_t lb;
                    if (!wait_slot(unit, lb)) return false;
                    fence_proxy_async();
                    fence_after();
                    {
                        const uint64_t ql = DK + (hb0 >> 4), xl = DK + (lb >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) mma_w(d_t, xl + 2 * kk, ql + 2 * kk, ID_QK, 1u, leader);
                    }
                    if (nheld == 2) {
                        const uint64_t ql = DK + (hb1 >> 4), xl = DK + ((lb + PAIR) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 4; kk++) mma_w(d_t, xl + 2 * kk, ql + 2 * kk, ID_QK, 1u, leader);
                    }
                    free_slot(hu0);
                    if (nheld == 2) free_slot(hu1);
                    free_slot(unit++);
                    nheld = 0;
                }
            }
            mma_commit_w(bar(B_SFULL0 + sb), leader);
            // every query chunk of this item has been read: its split buffer may be refilled
            if (last) mma_commit_w(bar(B_QFREE0 + (tok & 1)), leader);
            return true;
        };
        // O of tile i; `first`: the item's first tile (overwrites the accumulator), which
        // waits per d-block until the epilogue has read the previous item's block
        auto do_pv = [&](int i, bool first) -> bool {
            for (int j = 0; j < Lay::DB; j++) {
                if (first && tok > 0 && (j & 1) == 0) {
                    if (!wait_all(bar(B_OFREE0 + (j >> 1)), (tok - 1) & 1)) return false;
                    fence_after();
                }
                const uint32_t d_o = tmem + Lay::T_O + j * H;
                const bool has_lo = i == 0 || j >= p.nope_blocks;
                uint32_t xb;
                if (!wait_slot(unit, xb)) return false;
                fence_proxy_async();
                fence_after();
                // MN-major operands, 16 rows (128 descriptor units) per K step; rows 0 .. 63 in the
                // slot's first half, 64 .. 127 in its second
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const uint32_t aoff = (uint32_t)((kk >> 2) * PAIR + (kk & 3) * 2048);
                    const uint64_t ah = DA + ((xb + aoff) >> 4);
                    const uint64_t bh = DP + ((phi + kk * 2048) >> 4), bl = DP + ((plo + kk * 2048) >> 4);
                    mma_w(d_o, ah, bh, ID_PV, (first && kk == 0) ? 0u : 1u, leader);
                    mma_w(d_o, ah, bl, ID_PV, 1u, leader);
                }
                free_slot(unit++);
                if (has_lo) {
                    uint32_t lb;
                    if (!wait_slot(unit, lb)) return false;
                    fence_proxy_async();
                    fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; kk++) {
                        const uint32_t aoff = (uint32_t)((kk >> 2) * PAIR + (kk & 3) * 2048);
                        mma_w(d_o, DA + ((lb + aoff) >> 4), DP + ((phi + kk * 2048) >> 4), ID_PV, 1u, leader);
                    }
                    free_slot(unit++);
                }
            }
            mma_commit_w(bar(B_PVDONE), leader);
            return true;
        };
        const int n_items = p.n_q * p.parts;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Tok k = token_geom(p, it / p.parts);
            const int nc = comp_rows(p, k, nullptr);          // whole warp
            const Item itm = item_tiles(p, it, 1 + (nc + ROWS - 1) / ROWS);
            if (itm.tb >= itm.te) continue;
            bool good = do_qk(g, itm.tb, itm.tb == itm.te - 1);
            for (int i = itm.tb; i < itm.te && good; i++) {
                const uint32_t gi = g + (i - itm.tb);
                if (i + 1 < itm.te && !do_qk(gi + 1, i + 1, i + 1 == itm.te - 1)) { good = false; break; }
                if (!wait_all(bar(B_PFULL), gi & 1)) { good = false; break; }
                fence_after();
                if (!do_pv(i, i == itm.tb)) { good = false; break; }
            }
            ok = good;
            g += itm.te - itm.tb;
            tok++;
        }
        // drain: every MMA issued so far completes before the TMEM is freed (one more commit
        // tracks all of them; bounded, given up or not)
        if (lane == 0) {
            mma_commit(bar(B_DRAIN));
            mbar_drain(bar(B_DRAIN), 0);
        }
        __syncwarp();
    }
    } else if (warp < 8) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REG_SOFT));
        // ------------------------------------------------------------ softmax
        const int q4 = warp & 3;                 // TMEM lane quarter
        const int r = q4 * 32 + lane;            // tile row
        const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
        uint8_t *phi_p = sm + Lay::OFF_PHI;
        uint8_t *plo_p = sm + Lay::OFF_PLO;
        const int tid = threadIdx.x - 128;       // 0..127
        uint32_t g = 0, sphase = 0, tok = 0;
        bool ok = true;
        // barrier of the 128 softmax threads on an mbarrier, so that its wait is bounded
        auto soft_bar = [&]() -> bool {
            mbar_arrive(bar(B_SOFT));
            const bool r_ = mbar_wait(bar(B_SOFT), sphase, abort);
            sphase ^= 1;
            return r_;
        };
        const int n_items = p.n_q * p.parts;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const int n = it / p.parts;
            const Tok k = token_geom(p, n);
            const int nc = comp_rows(p, k, nullptr);
            const Item itm = item_tiles(p, it, 1 + (nc + ROWS - 1) / ROWS);
            if (itm.tb >= itm.te) {
                // empty part: no rows, zero weight in the combine
                if (tid < p.nh) {
                    p.part_ml[(size_t)it * 2 * p.nh + tid] = -INFINITY;
                    p.part_ml[(size_t)it * 2 * p.nh + p.nh + tid] = 0.f;
                }
                continue;
            }
            if (tid < H) mref_s[tid] = -INFINITY;
            // this lane's share of the softmax denominators (heads 2 lane, 2 lane + 1, the
            // warp's rows), rescaled with O whenever the reference maximum moves
            float lacc0 = 0.f, lacc1 = 0.f;
            if (!soft_bar()) { ok = false; break; }
            for (int i = itm.tb; i < itm.te; i++, g++) {
                const int sb = g & 1;
                if (!mbar_wait(bar(B_SFULL0 + sb), (g >> 1) & 1, abort)) { ok = false; break; }
                fence_after();
                float s[H];
                tmem_load_s<H>(lane_base + Lay::T_S + sb * 2 * H, s);
                fence_before();
                mbar_arrive(bar(B_SFREE0 + sb));
                const bool valid = (i == 0) ? (r >= k.raw_lo && r <= k.raw_hi) : ((i - 1) * ROWS + r < nc);
                bool need = false;
#pragma unroll
                for (int h = 0; h < H; h++) {
                    s[h] = valid ? s[h] * p.scale_log2 : -INFINITY;
                    need |= s[h] > mref_s[h] + TAU;
                }
                // block-wide vote among the 128 softmax threads
                const unsigned bal = __ballot_sync(0xffffffffu, need);
                if (lane == 0) flags[(g & 1) * 4 + q4] = bal ? 1 : 0;
                if (!soft_bar()) { ok = false; break; }
                const bool any = flags[(g & 1) * 4 + 0] | flags[(g & 1) * 4 + 1] | flags[(g & 1) * 4 + 2] |
                                 flags[(g & 1) * 4 + 3];
                bool waited = false;
                if (any) {
                    // exact tile maximum per head, then the new reference and the rescale factors.
                    // Warp maximum by a transposing butterfly: at offset o each lane keeps the
                    // half of its heads selected by lane bit o and takes the partner's maxima for
                    // it, so after the five steps lane l holds heads 2l and 2l + 1.
                    static_assert(H == 64, "the butterfly below assumes 64 heads");
                    float m[2];
                    warp_heads_reduce<true>(s, m[0], m[1]);
                    // the four warps' maxima meet in one key per head (the previous
                    // tile's factors have been read by now: the vote barrier came after)
                    if (tid < H) tmax[tid] = 0u;
                    if (!soft_bar()) { ok = false; break; }
                    atomicMax(&tmax[2 * lane], max_key(m[0]));
                    atomicMax(&tmax[2 * lane + 1], max_key(m[1]));
                    if (!soft_bar()) { ok = false; break; }
                    if (tid < H) {
                        const float mt = key_max(tmax[tid]);
                        const float mo = mref_s[tid];
                        const float mn = fmaxf(mo, mt);
                        alpha_s[tid] = exp2f(mo - mn);
                        mref_s[tid] = mn;
                    }
                    if (!soft_bar()) { ok = false; break; }
                    lacc0 *= alpha_s[2 * lane];
                    lacc1 *= alpha_s[2 * lane + 1];
                    if (i > itm.tb) {
                        if (!mbar_wait(bar(B_PVDONE), (g - 1) & 1, abort)) { ok = false; break; }
                        waited = true;
                        fence_after();
                        float v[H];
                        for (int j = 0; j < Lay::DB; j++) {
                            tmem_load<H>(lane_base + Lay::T_O + j * H, v);
#pragma unroll
                            for (int h = 0; h < H; h++) v[h] *= alpha_s[h];
                            tmem_store<H>(lane_base + Lay::T_O + j * H, v);
                        }
                        fence_before();
                    }
                }
                // the P buffers are free once the previous tile's O (of this item or the
                // previous one) has been computed
                if (g > 0 && !waited) {
                    if (!mbar_wait(bar(B_PVDONE), (g - 1) & 1, abort)) { ok = false; break; }
                }
                // P^T row r (MN-major, 128-byte swizzle), hi and lo
#pragma unroll
                for (int h = 0; h < H; h++) s[h] = exp2f(s[h] - mref_s[h]);
#pragma unroll
                for (int u = 0; u < H / 8; u++) {
                    float hv[8], lv[8];
#pragma unroll
                    for (int e = 0; e < 8; e++) split_bf16(s[u * 8 + e], hv[e], lv[e]);
                    const int off = r * (H * 2) + ((u ^ (r & 7)) * 16);
                    *reinterpret_cast<uint4 *>(phi_p + off) = make_uint4(pack_bf16x2(hv[0], hv[1]), pack_bf16x2(hv[2], hv[3]),
                                                                         pack_bf16x2(hv[4], hv[5]), pack_bf16x2(hv[6], hv[7]));
                    *reinterpret_cast<uint4 *>(plo_p + off) = make_uint4(pack_bf16x2(lv[0], lv[1]), pack_bf16x2(lv[2], lv[3]),
                                                                         pack_bf16x2(lv[4], lv[5]), pack_bf16x2(lv[6], lv[7]));
                }
                fence_proxy_async();
                mbar_arrive(bar(B_PFULL));
                {
                    float l0, l1;
                    warp_heads_reduce<false>(s, l0, l1);
                    lacc0 += l0;
                    lacc1 += l1;
                }
                if (i == itm.te - 1) {
                    // L[h] = (warp 0 + warp 1) + (warp 2 + warp 3) into the denominator words,
                    // warps 2 and 3 meeting in the tile-maximum words (once every warp is done
                    // with this tile's rescale factors there).  The denominator words still hold
                    // the previous item's L until its epilogue has read them (which precedes its
                    // first output-free arrival).
                    if (tok > 0 && !mbar_wait(bar(B_OFREE0), (tok - 1) & 1, abort)) { ok = false; break; }
                    if (!soft_bar()) { ok = false; break; }
                    float *lb = reinterpret_cast<float *>(tmax);
                    if (q4 == 0) { lfin[2 * lane] = lacc0; lfin[2 * lane + 1] = lacc1; }
                    if (q4 == 2) { lb[2 * lane] = lacc0; lb[2 * lane + 1] = lacc1; }
                    if (!soft_bar()) { ok = false; break; }
                    if (q4 == 1) { lfin[2 * lane] += lacc0; lfin[2 * lane + 1] += lacc1; }
                    if (q4 == 3) { lb[2 * lane] += lacc0; lb[2 * lane + 1] += lacc1; }
                    if (!soft_bar()) { ok = false; break; }
                    if (tid < H) {
                        const float l = lfin[tid] + lb[tid];
                        lfin[tid] = l;
                        // split rows: this part's reference maximum and denominator
                        if (p.parts > 1 && tid < p.nh) {
                            p.part_ml[(size_t)it * 2 * p.nh + tid] = mref_s[tid];
                            p.part_ml[(size_t)it * 2 * p.nh + p.nh + tid] = l;
                        }
                    }
                    mbar_arrive(bar(B_LREADY));
                }
            }
            tok++;
        }
    } else {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REG_AUX));
        // ------------------------------------------------------------ Q loader / epilogue
        const int q4 = warp & 3;                 // TMEM lane quarter
        const int r = q4 * 32 + lane;            // d within a 128-wide block
        const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
        const int tid = threadIdx.x - 256;       // 0..127
        uint32_t tok = 0, g = 0;
        bool ok = true;
        // fp32 Q [H][D] of the item's query, split into bf16 hi / lo, into this CTA's buffer
        // `buf` as D/64 query chunks [2H][64] (rows 0 .. H-1 hi, H .. 2H-1 lo), which the
        // producer loads by TMA into the 128-byte-swizzled K-major operand layout
        auto prepare = [&](int item, int buf) {
            if (p.qpre) {                                // split before the launch
                mbar_arrive(bar(B_QREADY0 + buf));
                return;
            }
            // heads past the layer's (nh < H) get zero query rows: their logits are 0 and their
            // outputs are not stored
            const float4 *src = reinterpret_cast<const float4 *>(p.q + (size_t)(item / p.parts) * p.q_ld);
            const int nf_real = p.nh * (D / 4);
            uint16_t *qd = p.qsplit + ((size_t)blockIdx.x * 2 + buf) * Lay::DC * 2 * H * 64;
            constexpr int NF = H * D / 4 / 128;           // float4 per thread
            static_assert(NF % 8 == 0, "whole batches of eight loads");
            for (int j0 = 0; j0 < NF; j0 += 8) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int f = tid + 128 * (j0 + u);
                    v[u] = f < nf_real ? __ldcs(src + f) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 8; u++) {
                    const int f = tid + 128 * (j0 + u);
                    const int h = f / (D / 4), d = (f % (D / 4)) * 4;
                    uint16_t *row = qd + ((size_t)(d / 64) * 2 * H + h) * 64 + (d % 64);
                    float h0, l0, h1, l1, h2, l2, h3, l3;
                    split_bf16(v[u].x, h0, l0);
                    split_bf16(v[u].y, h1, l1);
                    split_bf16(v[u].z, h2, l2);
                    split_bf16(v[u].w, h3, l3);
                    *reinterpret_cast<uint2 *>(row) = make_uint2(pack_bf16x2(h0, h1), pack_bf16x2(h2, h3));
                    *reinterpret_cast<uint2 *>(row + H * 64) = make_uint2(pack_bf16x2(l0, l1), pack_bf16x2(l2, l3));
                }
            }
            // the producer's TMA (async proxy) reads what these stores wrote
            asm volatile("fence.proxy.async.global;" ::: "memory");
            mbar_arrive(bar(B_QREADY0 + buf));
        };
        const int n_items = p.n_q * p.parts;
        int it = next_item(p, blockIdx.x, n_items);
        if (it < n_items) prepare(it, 0);
        while (ok && it < n_items) {
            const int nx = next_item(p, it + gridDim.x, n_items);
            const Tok k = token_geom(p, it / p.parts);
            const int nc = comp_rows(p, k, nullptr);
            const Item itm = item_tiles(p, it, 1 + (nc + ROWS - 1) / ROWS);
            const uint32_t nt = (uint32_t)(itm.te - itm.tb);
            // the next query into the other buffer, once the item that last used it (the
            // previous one) has had all its query chunks read
            if (nx < n_items) {
                const int nb = (tok + 1) & 1;
                if (tok >= 1 && !mbar_wait(bar(B_QFREE0 + nb), ((tok - 1) >> 1) & 1, abort)) { ok = false; break; }
                prepare(nx, nb);
            }
            // this item's output once its last O and its denominators are complete
            if (!mbar_wait(bar(B_LREADY), tok & 1, abort)) { ok = false; break; }
            if (!mbar_wait(bar(B_PVDONE), (g + nt - 1) & 1, abort)) { ok = false; break; }
            fence_after();
            // whole query: out[n][h][d] = O / L; split rows: the unnormalised partial part_o[it][h][d]
            const bool whole = p.parts == 1;
            float inv[H];
#pragma unroll
            for (int h = 0; h < H; h++) inv[h] = whole ? 1.0f / lfin[h] : 1.0f;
            float *dst = (whole ? p.out + (size_t)it * p.o_ld : p.part_o + (size_t)it * p.nh * D) + r;
            for (int j = 0; j < Lay::DB; j++) {
                float v[H];
                tmem_load<H>(lane_base + Lay::T_O + j * H, v);
                fence_before();
                if ((j & 1) || j == Lay::DB - 1) mbar_arrive(bar(B_OFREE0 + (j >> 1)));
#pragma unroll
                for (int h = 0; h < H; h++)
                    if (h < p.nh) __stcs(dst + (size_t)h * D + 128 * j, v[h] * inv[h]);
            }
            g += nt;
            tok++;
            it = nx;
        }
    }
    __syncthreads();
    if (warp == 1) {
        fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(Lay::T_COLS) : "memory");
    }
}

// Raw mirror: bf16 hi/lo of the raw rows in the order the kernel reads them.
// Prefill: row u <-> position pos0 - 128 + u (zeros before position 0), rows
// 0 .. 127 from the ring, the rest from raw_new.  Decode: sequence b owns rows
// 128b .. 128b+127 = its ring slots, with slot pos_b % 128 replaced by raw_new[b].
constexpr int SPLIT_ROWS = 4;             // mirror rows per block of raw_split_kernel

__global__ void raw_split_kernel(uint16_t *__restrict__ mirror, const float *__restrict__ ring,
                                 const float *__restrict__ raw_new, int D, int n_seq, int n_tok, uint64_t pos0,
                                 DecodePos dp, int n_rows, const float *__restrict__ q, uint16_t *__restrict__ qsplit,
                                 int nh, int64_t q_ld, int S, int early) {
    const int raw_blocks = (n_rows + SPLIT_ROWS - 1) / SPLIT_ROWS;
    if ((int)blockIdx.x >= raw_blocks) {
        // the query split (decode): one 64-d chunk c of query n per block, as the attention's
        // query chunks [2 x 64 heads][64] bf16 (hi rows, then lo rows; heads past nh zero).  Its
        // inputs are the call's own, so it runs before the wait for the previous kernel, which
        // it still takes before finishing (the dependent attention waits for this grid).
        const int DC = D / 64, qb = blockIdx.x - raw_blocks;
        const int n = qb / DC, c = qb % DC;
        uint16_t *qd = qsplit + ((size_t)n * DC + c) * 2 * 64 * 64;
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; k++) {                  // 64 heads x 16 float4, every load first
            const int f = threadIdx.x + 128 * k, h = f >> 4, e = (f & 15) * 4;
            v[k] = h < nh ? *reinterpret_cast<const float4 *>(q + (size_t)n * q_ld + (size_t)h * D + 64 * c + e)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 8; k++) {
            const int f = threadIdx.x + 128 * k, h = f >> 4, e = (f & 15) * 4;
            const float a4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            float hh[4], ll[4];
            for (int i = 0; i < 4; i++) split_bf16(a4[i], hh[i], ll[i]);
            *reinterpret_cast<uint2 *>(qd + (size_t)h * 64 + e) = make_uint2(pack_bf16x2(hh[0], hh[1]), pack_bf16x2(hh[2], hh[3]));
            *reinterpret_cast<uint2 *>(qd + (size_t)(64 + h) * 64 + e) =
                make_uint2(pack_bf16x2(ll[0], ll[1]), pack_bf16x2(ll[2], ll[3]));
        }
        pdl_launch_dependents();
        pdl_wait();
        return;
    }
    // early: the previous kernel writes neither the ring nor the mirror (the top-k or the decode
    // compressor), so the rows are split before the wait; the last block (and every query
    // block) still waits before finishing, so this grid completes only after that kernel
    if (!early) pdl_wait();
    pdl_launch_dependents();
    // the source row of mirror row u (null: zeros)
    auto source = [&](int u) -> const float * {
        if (n_seq == 1) {
            const int64_t pos = (int64_t)pos0 - ROWS + u;
            if (pos < 0 || pos < (int64_t)pos0 - S) return nullptr;  // before 0, or older than the ring holds
            return (pos < (int64_t)pos0) ? ring + (size_t)(pos % S) * D : raw_new + (size_t)(pos - (int64_t)pos0) * D;
        }
        const int b = u / ROWS, slot = u % ROWS;
        const uint64_t pos = dp.pos[b];
        if (slot >= S) return nullptr;                                // past the ring
        if (pos < (uint64_t)S && (uint64_t)slot > pos) return nullptr;  // slot not written yet
        return ((uint64_t)slot == pos % S) ? raw_new + (size_t)b * D : ring + ((size_t)b * S + slot) * D;
    };
    const int u0 = blockIdx.x * SPLIT_ROWS;
    for (int j = threadIdx.x * 4; j < D; j += blockDim.x * 4) {
        float4 v[SPLIT_ROWS];
#pragma unroll
        for (int r = 0; r < SPLIT_ROWS; r++) {           // every row's load before the first store
            const float *src = (u0 + r < n_rows) ? source(u0 + r) : nullptr;
            v[r] = src ? *reinterpret_cast<const float4 *>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int r = 0; r < SPLIT_ROWS; r++) {
            if (u0 + r >= n_rows) break;
            uint16_t *hi = mirror + (size_t)(u0 + r) * 2 * D;
            uint16_t *lo = hi + D;
            const float a4[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
            float h[4], l[4];
            for (int e = 0; e < 4; e++) split_bf16(a4[e], h[e], l[e]);
            *reinterpret_cast<uint2 *>(hi + j) = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
            *reinterpret_cast<uint2 *>(lo + j) = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
        }
    }
    if (early && (int)blockIdx.x == raw_blocks - 1) pdl_wait();
}

// Split rows: out = sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p over the
// parts of a query (M = the largest reference of a non-empty part).  Every
// thread reads its head's part maxima and denominators together with its
// partial outputs and forms the weights itself, so the block has no barrier.
constexpr int COMBINE_MAX_PARTS = 8;
__global__ void __launch_bounds__(128) attn_combine_kernel(float *__restrict__ out, int64_t o_ld,
                                                           const float *__restrict__ part_o,
                                                           const float *__restrict__ part_ml, int H, int D, int parts,
                                                           float *__restrict__ ring, const float *__restrict__ raw_new,
                                                           int S, DecodePos dp) {
    pdl_wait();
    pdl_launch_dependents();
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    // ring commit of the step (decode: query n is sequence n): the attention read the ring
    // through the raw mirror, so the slot can take the new row now
    if (ring && h == 0) {
        float *dst = ring + ((size_t)n * S + (size_t)(dp.pos[n] % (uint64_t)S)) * D;
        const float *src = raw_new + (size_t)n * D;
        for (int d = threadIdx.x * 4; d < D; d += blockDim.x * 4)
            *reinterpret_cast<float4 *>(dst + d) = *reinterpret_cast<const float4 *>(src + d);
    }
    for (int d = threadIdx.x * 4; d < D; d += blockDim.x * 4) {
        float m[COMBINE_MAX_PARTS], l[COMBINE_MAX_PARTS];
        float4 o[COMBINE_MAX_PARTS];
#pragma unroll
        for (int q = 0; q < COMBINE_MAX_PARTS; q++) {
            if (q >= parts) break;
            const float *ml = part_ml + ((size_t)n * parts + q) * 2 * H;
            m[q] = ml[h];
            l[q] = ml[H + h];
            o[q] = *reinterpret_cast<const float4 *>(part_o + (((size_t)n * parts + q) * H + h) * D + d);
        }
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < COMBINE_MAX_PARTS; q++)
            if (q < parts && l[q] > 0.f) M = fmaxf(M, m[q]);
        float den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < COMBINE_MAX_PARTS; q++) {
            if (q >= parts || !(l[q] > 0.f)) continue;
            const float wq = exp2f(m[q] - M);
            den += wq * l[q];
            acc.x += wq * o[q].x; acc.y += wq * o[q].y; acc.z += wq * o[q].z; acc.w += wq * o[q].w;
        }
        const float id = 1.0f / den;
        *reinterpret_cast<float4 *>(out + (size_t)n * o_ld + (size_t)h * D + d) =
            make_float4(acc.x * id, acc.y * id, acc.z * id, acc.w * id);
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

// 2-D bf16 map over `rows` rows of D elements with row pitch `pitch` bytes.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, int D, uint64_t pitch, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)pitch};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

template <int H, int D>
cudaError_t launch_hd(const AttnTcArgs &a, const TcAttnParams &p, bool commit, cudaStream_t s) {
    using Lay = L<H, D>;
    const uint64_t raw_rows = (a.n_seq == 1) ? (uint64_t)(ROWS + a.n_tok) : (uint64_t)a.n_seq * ROWS;
    CUtensorMap rh, rl;
    const uint64_t pitch = (uint64_t)2 * D * 2;
    if (!make_map(&rh, a.raw_mirror, raw_rows, D, pitch, 64) || !make_map(&rl, a.raw_mirror + D, raw_rows, D, pitch, 64))
        return cudaErrorNotSupported;
    const int items = a.n_seq * a.n_tok * p.parts;
    const int grid = items < sm_count() ? items : sm_count();
    // the split queries: per CTA two buffers of D/64 chunks [2H][64] bf16, one 128-row box each
    CUtensorMap qm;
    const uint64_t q_bufs = p.qpre ? (uint64_t)a.n_seq * a.n_tok : (uint64_t)grid * 2;
    if (!make_map(&qm, a.qsplit, q_bufs * Lay::DC * 2 * H, 64, 128, 2 * H)) return cudaErrorNotSupported;
    cudaError_t e = ensure_dyn_smem(attn_tc_kernel<H, D>, Lay::SMEM);
    if (e != cudaSuccess) return e;
    // the register reallocation at entry needs the launch allocation to cover both shares
    // (a shortfall would leave the softmax warpgroup waiting for registers): refuse otherwise
    static int regs = -1;
    if (regs < 0) {
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, attn_tc_kernel<H, D>);
        if (e != cudaSuccess) return e;
        regs = fa.numRegs;
    }
    if (4 * 32 * (REG_LOW + REG_SOFT + REG_AUX) > THREADS * regs) return cudaErrorNotSupported;
    e = launch_pdl(attn_tc_kernel<H, D>, dim3(grid), dim3(THREADS), Lay::SMEM, s, rh, rl, qm, p);
    if (e != cudaSuccess || p.parts == 1) return e;
    if (p.parts > COMBINE_MAX_PARTS) return cudaErrorNotSupported;
    return launch_pdl(attn_combine_kernel, dim3(a.n_seq * a.n_tok * p.nh), dim3(128), 0, s, p.out, p.o_ld,
                      (const float *)p.part_o, (const float *)p.part_ml, p.nh, D, p.parts,
                      commit ? const_cast<float *>(a.ring) : nullptr, a.raw_new, a.S, p.dp);
}

}  // namespace

size_t attn_tc_qsplit_bytes(int H, int D) {
    (void)H;                                           // the kernel always runs 64 heads
    return (size_t)sm_count() * 2 * 2 * 64 * D * sizeof(uint16_t);
}

int attn_tc_decode_parts(int ratio, int k, int comp_cap) {
    // the raw tile alone and about two compressed tiles per further work item: each item
    // loads its query's Q and writes one partial, so halving the item count against one
    // tile per item saves those fixed costs while a decode batch still spreads over the SMs
    const int rows = ratio == 4 ? (k < comp_cap ? k : comp_cap) : (ratio == 128 ? comp_cap : 0);
    const int tiles = 1 + (rows + ROWS - 1) / ROWS;
    const int parts = tiles == 1 ? 1 : 1 + tiles / 2;
    return parts < COMBINE_MAX_PARTS ? parts : COMBINE_MAX_PARTS;
}

bool attn_tc_supported(int H, int D, int S, int ratio, int k) {
    // 64 query heads per launch (fewer are padded to 64: the S product's N = 2H and the output
    // accumulator's H columns per d-block fill the 512 TMEM columns at 64); more than 64 run
    // as groups of 64
    const bool hd = H >= 1 && H <= 128 && (D == 512 || D == 256 || D == 128);
    // a raw window of at most one 128-row tile (a shorter one masks the tile's older rows)
    return hd && S >= 1 && S <= ROWS && (ratio == 0 || ratio == 4 || ratio == 128) && (ratio != 4 || k <= MAX_LIST);
}

cudaError_t launch_attention_tc(const AttnTcArgs &a, const DecodePos *dp, cudaStream_t s) {
    const int nq = a.n_seq * a.n_tok;
    if (nq <= 0) return cudaSuccess;
    DecodePos dd{};
    if (a.n_seq > 1) dd = *dp;
    const int raw_rows = (a.n_seq == 1) ? ROWS + a.n_tok : a.n_seq * ROWS;
    // split rows (decode): the queries are split here, by many blocks, instead of by each work
    // item's CTA on its critical path; the per-CTA query buffers hold 2 x sm_count queries
    const int parts = a.parts > 0 ? a.parts : 1;
    const bool qpre = parts > 1 && nq <= 2 * sm_count();
    const int q_blocks = qpre ? nq * (a.D / 64) : 0;
    // More than 64 heads run as groups of 64 (the last one padded), one raw split, attention
    // and (split rows) combine per group, each over the same rows; the ring takes the step's
    // row after the last group (the combine) or after the call (ring commit)
    const int groups = (a.H + 63) / 64;
    for (int g = 0; g < groups; g++) {
        const int h0 = 64 * g, nh = a.H - h0 < 64 ? a.H - h0 : 64;
        const float *q = a.q + (size_t)h0 * a.D;
        // raw mirror (and, split rows, the queries of this group)
        const int early = (pdl_prev_is(s, PDL_TOPK) || pdl_prev_is(s, PDL_DECODE_COMPRESS)) ? 1 : 0;
        cudaError_t e = launch_pdl(raw_split_kernel, dim3((raw_rows + SPLIT_ROWS - 1) / SPLIT_ROWS + q_blocks),
                                   dim3(128), 0, s, a.raw_mirror, a.ring, a.raw_new, a.D, a.n_seq, a.n_tok, a.pos0, dd,
                                   raw_rows, q, a.qsplit, nh, (int64_t)a.H * a.D, a.S, early);
        if (e != cudaSuccess) return e;
        TcAttnParams p{};
        p.out = a.out + (size_t)h0 * a.D;
        p.q = q;
        p.q_ld = p.o_ld = (int64_t)a.H * a.D;
        p.nh = nh;
        p.qsplit = a.qsplit;
        p.qpre = qpre ? 1 : 0;
        p.topk = a.topk;
        p.comp_split = a.comp_split;
        p.nope_chunks = (a.D - a.n_rot) / 64;
        p.nope_blocks = (a.D - a.n_rot) / 128;
        p.parts = parts;
        p.part_o = a.part_o;
        p.part_ml = a.part_ml;
        p.n_q = nq;
        p.n_seq = a.n_seq;
        p.n_tok = a.n_tok;
        p.k = a.k;
        p.ratio = a.ratio;
        p.comp_cap = a.comp_cap;
        p.swa = a.S;
        p.scale_log2 = a.scale * 1.4426950408889634f;
        p.pos0 = a.pos0;
        p.dp = dd;
        const bool commit = a.commit_ring && g == groups - 1;
        e = cudaErrorNotSupported;
        if (a.D == 512) e = launch_hd<64, 512>(a, p, commit, s);
        else if (a.D == 256) e = launch_hd<64, 256>(a, p, commit, s);
        else if (a.D == 128) e = launch_hd<64, 128>(a, p, commit, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t attn_tc_set_wait_ns(unsigned long long ns) { return cudaMemcpyToSymbol(g_attn_wait_ns, &ns, sizeof ns); }

unsigned int attn_tc_read_clear_error() {
    unsigned int v = 0, z = 0;
    if (cudaMemcpyFromSymbol(&v, g_attn_tc_err, sizeof v) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_attn_tc_err, &z, sizeof z);
    return v;
}

}  // namespace ds4c
