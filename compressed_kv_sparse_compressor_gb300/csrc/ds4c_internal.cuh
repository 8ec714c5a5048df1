// Internal declarations of libds4c: kernel argument blocks and launchers.
// Every translation unit of the library includes this header; nothing outside
// the library does.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ds4c.h"

namespace ds4c {

constexpr int kMaxRot = 128;
constexpr int kMaxDecodeSeq = 1024;
constexpr uint32_t kMaxIdxCap = 40960;

// Host validation of a layer configuration (DS4C_OK or the status every call returns for it).
ds4c_status check_cfg(const ds4c_layer_cfg *c);
// DS4C_OK for cudaSuccess; otherwise records e for ds4c_last_cuda_error and returns DS4C_ERR_CUDA.
ds4c_status cuda_status(cudaError_t e);

inline int lane_width(const ds4c_layer_cfg &c, bool attn) { return attn ? (int)c.head_dim : (int)c.idx_head_dim; }
inline int coff_of(const ds4c_layer_cfg &c) { return c.ratio == 4 ? 2 : 1; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Opt a kernel into `bytes` of dynamic shared memory.  The default limit of
// 48 KiB covers static and dynamic shared memory together, so the opt-in is
// made for any request above 16 KiB (every kernel here has less than 16 KiB
// of static shared memory).  On failure the error is also taken out of the
// runtime's last-error slot, so it is reported once, by the caller.
template <typename F>
inline cudaError_t ensure_dyn_smem(F *func, size_t bytes) {
    if (bytes <= 16 * 1024) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

// Bounded waits.  Every spin of the kernels gives up after a limit (4 s), raises
// its translation unit's device error word and winds the CTA down; the limit
// sits in a device variable of each unit, changed only by the test hook
// ds4c_test_set_wait_limit.  Waits that drain copies or MMAs still in flight
// after a give-up use kDrainNs whatever that limit is.
constexpr unsigned long long kWaitNsDefault = 4000000000ull;
constexpr unsigned long long kDrainNs = 4000000000ull;
cudaError_t gemm_tc_set_wait_ns(unsigned long long ns);
cudaError_t attn_tc_set_wait_ns(unsigned long long ns);
cudaError_t idx_set_wait_ns(unsigned long long ns);
// One CTA waits on an mbarrier that nothing arrives on, bounded by limit_ns, with
// the indexer kernels' wait routine: it gives up, raises the indexer's error word
// and returns (the self-test of the error path; no fault, no hang).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);

// FP32 FMA-rate probe (the ALU roofline's denominator): flops of one launch
// of `blocks` 256-thread CTAs running `iters` rounds, and the launch itself.
double fma_probe_flops(uint32_t blocks, uint32_t iters);
cudaError_t launch_fma_probe(uint32_t blocks, uint32_t iters, float *out, cudaStream_t s);

// Programmatic dependent launch.  Kernels launched by launch_pdl may be
// scheduled while the previous kernel of the stream is still finishing, so
// every such kernel calls pdl_wait() in each CTA before its first access to
// global memory written by the previous kernel, and before it exits: it returns
// once the previous kernel has completed and its writes are visible, which also
// orders every earlier kernel.  pdl_launch_dependents() lets the next kernel be
// scheduled.  Under an ordinary launch both are no-ops.  (The decode indexer
// score reads rows older than the newest before its wait when the previous
// kernel is the decode compressor, and the attention's raw-row split reads the
// ring before its wait when the previous kernel is the top-k or the decode
// compressor, see PdlPrev; its split query blocks read only the call's own
// inputs before theirs.)
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Indexer QAT round trip of one row held by G consecutive threads, four values
// each (element 4t + e in thread t of the group, e = x, y, z, w): the
// orthonormal Sylvester Hadamard transform evaluated as the binary32 fast
// Walsh-Hadamard butterfly (stage h combines x[j], x[j + h] with j & h == 0
// into x[j] + x[j + h], x[j] - x[j + h]) and one multiply by c = binary32(1 /
// sqrt(4G)), then an FP4 E2M1 round trip with one power-of-two scale per block
// of 32 values ("Metal グラフと圧縮 KV の実装を読む" §9: Hadamard 128 and FP4 on the
// indexer row and queries; the evaluation order, block and scale rule are this
// library's reading).  G <= 32, the group aligned inside its warp; every lane
// of the warp calls this.
// ----------------------------------------------------------------------------
// Nearest E2M1 value (0, 0.5, 1, 1.5, 2, 3, 4, 6) to y, ties to the even code,
// saturating at +-6; the sign of y is kept.
__device__ __forceinline__ float e2m1_rne(float y) {
    const float a = fabsf(y);
    float r;
    if (a <= 0.25f) r = 0.0f;          // 0.25: tie between codes 0 and 1 -> 0
    else if (a < 0.75f) r = 0.5f;      // 0.75: tie -> 1.0 (code 2)
    else if (a <= 1.25f) r = 1.0f;     // 1.25: tie -> 1.0 (code 2)
    else if (a < 1.75f) r = 1.5f;      // 1.75: tie -> 2.0 (code 4)
    else if (a <= 2.5f) r = 2.0f;      // 2.5: tie -> 2.0 (code 4)
    else if (a < 3.5f) r = 3.0f;       // 3.5: tie -> 4.0 (code 6)
    else if (a <= 5.0f) r = 4.0f;      // 5.0: tie -> 4.0 (code 6)
    else r = 6.0f;
    return copysignf(r, y);
}

// Smallest e with amax <= 6 * 2^e (0 for amax == 0).  With amax = m * 2^E,
// m in [0.5, 1): 6 * 2^(E-3) = 0.75 * 2^E, so e = E - 3 when m <= 0.75, else E - 2.
__device__ __forceinline__ int fp4_scale_exp(float amax) {
    if (!(amax > 0.f)) return 0;
    int E;
    const float m = frexpf(amax, &E);                     // exact
    return (m <= 0.75f) ? E - 3 : E - 2;
}

template <int G>
__device__ __forceinline__ void indexer_qat_group(float4 &v, float c) {
    static_assert(G >= 8 && G <= 32 && (G & (G - 1)) == 0, "QAT groups of 8 .. 32 threads");
    const int t = threadIdx.x % G;
    // stages h = 1 and 2 inside the thread
    float a0 = v.x + v.y, a1 = v.x - v.y, a2 = v.z + v.w, a3 = v.z - v.w;
    v = make_float4(a0 + a2, a1 + a3, a0 - a2, a1 - a3);
    // stages h = 4 .. 2G across threads: partner t ^ (h / 4)
#pragma unroll
    for (int o = 1; o < G; o <<= 1) {
        const float4 p = make_float4(__shfl_xor_sync(0xffffffffu, v.x, o), __shfl_xor_sync(0xffffffffu, v.y, o),
                                     __shfl_xor_sync(0xffffffffu, v.z, o), __shfl_xor_sync(0xffffffffu, v.w, o));
        if ((t & o) == 0) v = make_float4(v.x + p.x, v.y + p.y, v.z + p.z, v.w + p.w);
        else v = make_float4(p.x - v.x, p.y - v.y, p.z - v.z, p.w - v.w);
    }
    v = make_float4(v.x * c, v.y * c, v.z * c, v.w * c);
    // FP4: a block of 32 values is 8 consecutive threads
    float am = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const int e = fp4_scale_exp(am);
    v.x = ldexpf(e2m1_rne(ldexpf(v.x, -e)), e);
    v.y = ldexpf(e2m1_rne(ldexpf(v.y, -e)), e);
    v.z = ldexpf(e2m1_rne(ldexpf(v.z, -e)), e);
    v.w = ldexpf(e2m1_rne(ldexpf(v.w, -e)), e);
}

// What the kernel launch_pdl issued last on this thread (and its stream) writes, when a kernel
// launched right after it may read other data before waiting for it: set by the launchers of
// the decode compressor (which writes no compressed row but the newest of each sequence, and
// no raw ring, raw mirror or query) and of the top-k (which writes the row lists alone); any
// other launch clears it.  A caller's kernel in between is an ordinary launch, which the next
// kernel waits for in full.
enum PdlKind { PDL_ANY = 0, PDL_DECODE_COMPRESS = 1, PDL_TOPK = 2 };
struct PdlPrev {
    cudaStream_t s = nullptr;
    int kind = PDL_ANY;
};
inline PdlPrev &pdl_prev() {
    static thread_local PdlPrev v;
    return v;
}
inline bool pdl_prev_is(cudaStream_t s, int kind) { return pdl_prev().s == s && pdl_prev().kind == kind; }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    pdl_prev().kind = PDL_ANY;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// ----------------------------------------------------------------------------
// Projection GEMM: C[g][m][n] = sum_k A[m][k] * B[g][n][k], fp32 out.
// ----------------------------------------------------------------------------
struct GemmGroup {
    const void *B;      // [N][K] row-major, dtype
    float *C;           // [M][ldc]
    int64_t ldc;
    int N;
};
struct GemmArgs {
    const void *A;      // [M][K] row-major, dtype
    int M, K;
    int dtype;          // DS4C_F32 / DS4C_BF16
    int n_groups;
    GemmGroup g[4];
    // Optional split-K (tensor-core path): every group's C lies in one block
    // [M][part_ld] starting at c_base; part holds max_ksplit such blocks.
    float *c_base = nullptr;
    float *part = nullptr;
    int64_t part_ld = 0;
    int max_ksplit = 1;
    // Optional (tensor-core path, no split-K): room for gemm_tail_floats() floats, where the
    // output tiles of a last, partly filled round over the SMs are computed split along K
    float *tail_buf = nullptr;
};
// Floats of the GEMM's tail buffer (one 128 x 256 fp32 tile per SM).
size_t gemm_tail_floats();
cudaError_t launch_gemm_simt(const GemmArgs &a, cudaStream_t s);
// tcgen05 path for bf16 operands; returns cudaErrorNotSupported when the
// shape is outside what it handles (the caller then uses the SIMT kernel).
cudaError_t launch_gemm_tc(const GemmArgs &a, cudaStream_t s);
unsigned int gemm_tc_read_clear_error();

// ----------------------------------------------------------------------------
// Compressor (store + APE, pool, RMSNorm, tail RoPE, FP8, append, frontier).
// ----------------------------------------------------------------------------
struct RopeTable { float inv_freq[kMaxRot / 2]; };

struct LaneArgs {
    const float *kv;  int64_t kv_ld;   // projection output rows (kv part), [rows][ld]
    const float *sc;  int64_t sc_ld;   // projection output rows (score part)
    const float *ape;                  // [ratio][W]
    const float *gain;                 // [Dl] or null
    float *comp;                       // [n_seq][cap][Dl]
    float *prequant;                   // same or null
    float *skv, *ssc;                  // [n_seq][coff*ratio][W]
    uint16_t *split;                   // attention lane: [n_seq][cap][2][Dl] bf16 hi, lo (or null)
    int Dl, cap, is_attn;
    int qat;                           // indexer lane: Hadamard + FP4 round trip of each appended row
    float qat_c;                       // binary32(1 / sqrt(Dl)) of that round trip
};
struct CompressArgs {
    LaneArgs lane[2];
    int n_lanes;
    int ratio, n_rot;
    float eps;
    RopeTable rope;
    // segments: prefill = one segment (seq 0); decode = one token per sequence
    int n_seg;
    uint64_t pos0;        // prefill
    uint32_t T;           // prefill tokens
    const uint64_t *pos_d; // unused
};
struct DecodePos { uint64_t pos[kMaxDecodeSeq]; };

cudaError_t launch_compress_prefill(const CompressArgs &a, cudaStream_t s);
cudaError_t launch_compress_decode(const CompressArgs &a, const DecodePos &p, int n_seq, cudaStream_t s);

// ----------------------------------------------------------------------------
// Indexer score + top-k
// ----------------------------------------------------------------------------
struct IndexerArgs {
    const float *q;          // [n][d]
    const float *rows;       // [n_seq][idx_cap][d]
    int64_t seq_stride;      // idx_cap * d
    float *scores;           // [n][lds]
    int64_t lds;
    int32_t *topk;           // [n][k]
    int d, k;
    int n_seq, n_tok;
    uint64_t pos0;           // prefill
};
cudaError_t launch_indexer_prefill(const IndexerArgs &a, cudaStream_t s);
// Multi-head score (heads > 1, or one head with the ReLU-weighted form): q holds
// the heads' query vectors [n][heads][d] (after the round trip), w [n][heads];
// then the same top-k.  dp == nullptr for a prefill chunk of one sequence.
cudaError_t launch_indexer_heads(const IndexerArgs &a, const float *w, int heads, const DecodePos *dp, cudaStream_t s);
// Hadamard + FP4 round trip of n_vec vectors of d floats (d = 64 or 128), in -> out.
cudaError_t launch_qat_vectors(const float *in, float *out, int64_t n_vec, int d, float c, cudaStream_t s);
cudaError_t launch_indexer_decode(const IndexerArgs &a, const DecodePos &p, cudaStream_t s);
// device error word of the indexer kernels (a bounded wait gave up); read and cleared
unsigned int idx_read_clear_error();

// ----------------------------------------------------------------------------
// Sparse SWA attention + ring commit
// ----------------------------------------------------------------------------
struct AttnArgs {
    const float *q;          // [n][H][D]
    const float *raw_new;    // [n][D]
    const float *ring;       // [n_seq][S][D]
    const float *comp;       // [n_seq][comp_cap][D]
    const int32_t *topk;     // [n][k] or null
    float *out;              // [n][H][D]
    int D, H, S, ratio, k, comp_cap;
    float scale;
    int n_seq, n_tok;
    uint64_t pos0;
};
cudaError_t launch_attention(const AttnArgs &a, const DecodePos *p, cudaStream_t s);

// Tensor-core attention (H = 64, D in {128, 256, 512}, swa = 128).
struct AttnTcArgs {
    const float *q;
    const float *raw_new;
    const float *ring;
    const uint16_t *comp_split;   // [n_seq_state][comp_cap][2][D]
    uint16_t *raw_mirror;         // workspace: [rows][2][D]
    uint16_t *qsplit;             // workspace: attn_tc_qsplit_bytes
    const int32_t *topk;
    float *out;
    int D, H, ratio, k, comp_cap, n_rot;
    int S;                        // raw window = ring rows (at most 128)
    float scale;
    int n_seq, n_tok, n_seq_state;
    uint64_t pos0;
    int parts;                    // work items per query; > 1 splits the rows (decode)
    int commit_ring;              // parts > 1: the combine also writes raw_new[b] to ring slot pos_b % 128
    float *part_o, *part_ml;      // workspace for the partial outputs when parts > 1
};
// Work items per decode query: one per two 128-row tiles (the raw window plus
// the compressed rows a query can see), at most 8.
int attn_tc_decode_parts(int ratio, int k, int comp_cap);
// Workspace bytes of the split queries (two buffers per CTA, one CTA per SM).
size_t attn_tc_qsplit_bytes(int H, int D);
bool attn_tc_supported(int H, int D, int S, int ratio, int k);
cudaError_t launch_attention_tc(const AttnTcArgs &a, const DecodePos *p, cudaStream_t s);
unsigned int attn_tc_read_clear_error();
cudaError_t launch_ring_commit(float *ring, const float *raw_new, int D, int S, int n_seq, int n_tok,
                               uint64_t pos0, const DecodePos *p, cudaStream_t s);

// ----------------------------------------------------------------------------
// State init, checkpoint gather
// ----------------------------------------------------------------------------
cudaError_t launch_fill(float *p, size_t n, float v, cudaStream_t s);

struct GatherSeg { const float *src; int64_t dst_off; int64_t n; };
struct GatherArgs {
    float *dst;
    const float *ring; int64_t D; int64_t S; uint64_t pos; int64_t n_live;
    int n_seg;
    GatherSeg seg[8];
};
cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s);

// Restore (the gather's inverse): segment 0 writes the raw rows back to their
// ring slots, the others are contiguous copies from src + src_off.
struct ScatterSeg { float *dst; int64_t src_off; int64_t n; };
struct ScatterArgs {
    const float *src;
    float *ring; int64_t D; int64_t S; uint64_t pos; int64_t n_live;
    int n_seg;
    ScatterSeg seg[8];
};
cudaError_t launch_scatter(const ScatterArgs &a, cudaStream_t s);
// bf16 hi / lo of n_rows rows of D floats (the tensor-core attention's mirror)
cudaError_t launch_split_rows(uint16_t *split, const float *rows, int64_t n_rows, int D, cudaStream_t s);

}  // namespace ds4c
