// Fused compressor (K2): store + APE, boundary softmax pool, RMSNorm, tail
// RoPE, FP8 E4M3 round trip and append, for every compressed row a prefill
// chunk (or a decode step) completes; then the frontier commit (K2b) that
// leaves state_kv / state_score exactly as the token-by-token recurrence of
// "Metal グラフと圧縮 KV の実装を読む" §4-§5 would.
//
// The pages' Metal design runs store, pool and shift as separate dispatches per
// token (kernel_dsv4_compressor_store_one, kernel_dsv4_softmax_pool,
// kernel_dsv4_ratio4_shift_f32).  Here a chunk is processed at once: a row's
// pooling candidates are read straight from the projection output (or, for
// tokens before the chunk, from the frontier), so every kv / score element is
// read from HBM exactly once and the frontier is written once per chunk.
//
// Thread layout: a group of G = Dl/4 threads owns one compressed row, each
// thread a float4 column slice; a 128-thread block holds 128/G rows (ratio 4)
// or one row with 4 row-splits of the 128-token window (ratio 128).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ds4c_internal.cuh"

namespace ds4c {
namespace {

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ float4 add4(float4 a, float4 b) { return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); }
__device__ __forceinline__ float4 max4(float4 a, float4 b) {
    return make_float4(fmaxf(a.x, b.x), fmaxf(a.y, b.y), fmaxf(a.z, b.z), fmaxf(a.w, b.w));
}

// One pooling candidate of window c: token p of the chunk (projection output,
// score + APE row p % ratio) or, for p < pos0, the frontier row `srow`.
__device__ __forceinline__ void fetch(const LaneArgs &L, const float *skv, const float *ssc, int W, int ratio,
                                      int64_t p, int srow, int col, uint64_t pos0, int64_t ws_row0,
                                      float4 &kv, float4 &s) {
    if (p >= (int64_t)pos0) {
        int64_t row = ws_row0 + (p - (int64_t)pos0);
        kv = ld4(L.kv + row * L.kv_ld + col);
        s = add4(ld4(L.sc + row * L.sc_ld + col), ld4(L.ape + (size_t)(p % ratio) * W + col));
    } else {
        kv = ld4(skv + (size_t)srow * W + col);
        s = ld4(ssc + (size_t)srow * W + col);
    }
}

template <int G>
__device__ __forceinline__ float group_sum(float v, float *red) {
    // G threads, aligned inside the block.  G <= 32: shuffles inside the warp.
    if constexpr (G <= 32) {
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
        const int wpg = G / 32;                          // warps per group
        if (lane == 0) red[warp] = v;
        __syncthreads();
        float t = 0.f;
        const int g0 = (warp / wpg) * wpg;
        for (int w = 0; w < wpg; w++) t += red[g0 + w];
        __syncthreads();
        return t;
    }
}

// Smallest e with amax <= 448 * 2^e (0 for amax == 0): the block scale of the
// E4M3 round trip is the power of two 2^e ("Metal グラフと圧縮 KV の実装を読む" §9;
// the block size and scale rule are this library's reading).
__device__ __forceinline__ int fp8_scale_exp(float amax) {
    if (!(amax > 0.f)) return 0;
    int E;
    frexpf(amax, &E);                                   // amax = m * 2^E, m in [0.5, 1)
    return (amax <= ldexpf(448.f, E - 9)) ? E - 9 : E - 8;
}

__device__ __forceinline__ float e4m3_roundtrip(float y) {
    __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3);
    __half_raw h = __nv_cvt_fp8_to_halfraw(q, __NV_E4M3);
    return __half2float(__half(h));
}

// What a row's finish needs besides the pooled values: the RMSNorm gain of the
// thread's columns and, in the rotated tail, the sine and cosine of its two
// pairs' angles (both depend only on the row position and the columns, so they
// are fetched and computed before the pool, while its loads are in flight).
struct RowPrep {
    float4 g;
    float s0, c0, s1, c1;
};

__device__ __forceinline__ RowPrep row_prep(const CompressArgs &a, const LaneArgs &L, uint64_t c, int j) {
    RowPrep r;
    r.g = L.gain ? ld4(L.gain + j) : make_float4(1.f, 1.f, 1.f, 1.f);
    r.s0 = r.s1 = 0.f;
    r.c0 = r.c1 = 1.f;
    const int nope = L.Dl - a.n_rot;
    if (j >= nope) {
        const int i0 = (j - nope) / 2;
        const float pc = (float)(c * (uint64_t)a.ratio);
        sincosf(__fmul_rn(pc, a.rope.inv_freq[i0]), &r.s0, &r.c0);
        sincosf(__fmul_rn(pc, a.rope.inv_freq[i0 + 1]), &r.s1, &r.c1);
    }
    return r;
}

// RMSNorm -> tail RoPE -> (attention lane) FP8, then append.  x is this
// thread's float4 of the pooled row; all G threads of the group call this.
template <int G>
__device__ __forceinline__ void finish_row(const CompressArgs &a, const LaneArgs &L, bool active, int seq,
                                           uint64_t c, int j, float4 x, float *red, const RowPrep &rp) {
    const int Dl = L.Dl;
    float ss = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    ss = group_sum<G>(active ? ss : 0.f, red);
    const float inv = 1.0f / sqrtf(ss / (float)Dl + a.eps);
    const float4 g = rp.g;
    float4 y = make_float4(x.x * inv * g.x, x.y * inv * g.y, x.z * inv * g.z, x.w * inv * g.w);
    const int nope = Dl - a.n_rot;
    if (j >= nope) {
        float4 r;
        r.x = y.x * rp.c0 - y.y * rp.s0;
        r.y = y.x * rp.s0 + y.y * rp.c0;
        r.z = y.z * rp.c1 - y.w * rp.s1;
        r.w = y.z * rp.s1 + y.w * rp.c1;
        y = r;
    }
    const size_t off = ((size_t)seq * L.cap + (size_t)c) * Dl + j;
    if (active && L.prequant) st4(L.prequant + off, y);
    if constexpr (G >= 8 && G <= 32) {
        // indexer lane: Hadamard + FP4 round trip of the whole row ("Metal グラフと圧縮 KV の実装を読む" §9)
        if (!L.is_attn && L.qat) indexer_qat_group<G>(y, L.qat_c);
    }
    if (L.is_attn) {
        float am = (j < nope) ? fmaxf(fmaxf(fabsf(y.x), fabsf(y.y)), fmaxf(fabsf(y.z), fabsf(y.w))) : 0.f;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
        if (j < nope) {
            const int e = fp8_scale_exp(am);
            y.x = ldexpf(e4m3_roundtrip(ldexpf(y.x, -e)), e);
            y.y = ldexpf(e4m3_roundtrip(ldexpf(y.y, -e)), e);
            y.z = ldexpf(e4m3_roundtrip(ldexpf(y.z, -e)), e);
            y.w = ldexpf(e4m3_roundtrip(ldexpf(y.w, -e)), e);
        }
    }
    if (active) {
        st4(L.comp + off, y);
        if (L.split) {
            // bf16 hi / lo mirror of the appended row for the tensor-core attention
            const __nv_bfloat162 h01 = __floats2bfloat162_rn(y.x, y.y), h23 = __floats2bfloat162_rn(y.z, y.w);
            const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
            const __nv_bfloat162 l01 = __floats2bfloat162_rn(y.x - f01.x, y.y - f01.y);
            const __nv_bfloat162 l23 = __floats2bfloat162_rn(y.z - f23.x, y.w - f23.y);
            uint16_t *row = L.split + ((size_t)seq * L.cap + (size_t)c) * 2 * Dl;
            uint2 hv, lv;
            hv.x = *reinterpret_cast<const uint32_t *>(&h01);
            hv.y = *reinterpret_cast<const uint32_t *>(&h23);
            lv.x = *reinterpret_cast<const uint32_t *>(&l01);
            lv.y = *reinterpret_cast<const uint32_t *>(&l23);
            *reinterpret_cast<uint2 *>(row + j) = hv;
            *reinterpret_cast<uint2 *>(row + Dl + j) = lv;
        }
    }
}

// Softmax pool of a ratio-4 window's eight candidates, per column: the weights
// exp(s - max) over the eight, their sum as the denominator.
__device__ __forceinline__ float4 pool8(const float4 (&kv)[8], const float4 (&s)[8]) {
    float4 m = s[0];
#pragma unroll
    for (int q = 1; q < 8; q++) m = max4(m, s[q]);
    float4 den = make_float4(0.f, 0.f, 0.f, 0.f), sum = den;
#pragma unroll
    for (int q = 0; q < 8; q++) {
        float4 w = make_float4(expf(s[q].x - m.x), expf(s[q].y - m.y), expf(s[q].z - m.z), expf(s[q].w - m.w));
        den = add4(den, w);
        sum.x += w.x * kv[q].x; sum.y += w.y * kv[q].y; sum.z += w.z * kv[q].z; sum.w += w.w * kv[q].w;
    }
    float4 x;
    x.x = den.x > 0.f ? sum.x / den.x : 0.f;
    x.y = den.y > 0.f ? sum.y / den.y : 0.f;
    x.z = den.z > 0.f ? sum.z / den.z : 0.f;
    x.w = den.w > 0.f ? sum.w / den.w : 0.f;
    return x;
}

// Ratio 4: window c pools, per column j, rows 0..3 (previous window, columns
// [0, Dl)) and rows 4..7 (current window, columns [Dl, 2Dl)).
// One pooling task per G threads of a 128-thread block (decode: task = the
// sequence; prefill: the window index from pos0); every thread of the block
// calls this.
template <int G>
__device__ __forceinline__ void pool_r4(const CompressArgs &a, int lane_id, const DecodePos &dp, int decode, int task,
                                        float *red) {
    const LaneArgs L = a.lane[lane_id];
    const int W = 2 * L.Dl;
    const int j = (threadIdx.x % G) * 4;
    int seq = 0;
    uint64_t pos0, c;
    uint32_t T;
    int64_t ws_row0 = 0;
    bool active;
    if (decode) {
        seq = task;
        active = task < a.n_seg;
        pos0 = active ? dp.pos[task] : 0;
        T = 1;
        ws_row0 = task;
        c = pos0 / 4;
        active = active && ((pos0 + 1) % 4 == 0);
    } else {
        pos0 = a.pos0;
        T = a.T;
        c = pos0 / 4 + (uint64_t)task;
        active = c < (pos0 + T) / 4;
    }
    const float *skv = L.skv + (size_t)seq * 8 * W;
    const float *ssc = L.ssc + (size_t)seq * 8 * W;
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    RowPrep rp{};
    if (active) {
        float4 kv[8], s[8];
        const uint64_t cur = pos0 / 4;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int64_t p = 4 * ((int64_t)c - 1) + q;
            const int srow = (p < 0) ? q : (((uint64_t)p / 4 == cur) ? 4 + q : q);
            fetch(L, skv, ssc, W, 4, p, srow, j, pos0, ws_row0, kv[q], s[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int64_t p = 4 * (int64_t)c + q;
            fetch(L, skv, ssc, W, 4, p, 4 + q, L.Dl + j, pos0, ws_row0, kv[4 + q], s[4 + q]);
        }
        rp = row_prep(a, L, c, j);
        x = pool8(kv, s);
    }
    finish_row<G>(a, L, active, seq, c, j, x, red, rp);
}

template <int G>
__global__ void __launch_bounds__(128) compress_r4_kernel(CompressArgs a, int lane_id, DecodePos dp, int decode) {
    __shared__ float red[32];
    pdl_wait();
    pdl_launch_dependents();
    pool_r4<G>(a, lane_id, dp, decode, blockIdx.x * (128 / G) + threadIdx.x / G, red);
}

// Ratio 128: window c pools rows 0..127 at column j.  NS row-splits of the
// window run an online softmax each and are merged through shared memory.
template <int G>
__global__ void __launch_bounds__(G * 4) compress_r128_kernel(CompressArgs a, int lane_id, DecodePos dp, int decode) {
    constexpr int NS = 4;
    __shared__ float4 part[3][NS][G];
    __shared__ float red[32];
    pdl_wait();
    pdl_launch_dependents();
    const LaneArgs L = a.lane[lane_id];
    const int W = L.Dl;
    const int split = threadIdx.x / G;
    const int t = threadIdx.x % G;
    const int j = t * 4;
    int seq = 0;
    uint64_t pos0, c;
    uint32_t T;
    int64_t ws_row0 = 0;
    bool active;
    if (decode) {
        seq = blockIdx.x;
        active = seq < a.n_seg;
        pos0 = active ? dp.pos[seq] : 0;
        T = 1;
        ws_row0 = seq;
        c = pos0 / 128;
        active = active && ((pos0 + 1) % 128 == 0);
    } else {
        pos0 = a.pos0;
        T = a.T;
        c = pos0 / 128 + blockIdx.x;
        active = c < (pos0 + T) / 128;
    }
    (void)T;
    const float *skv = L.skv + (size_t)seq * 128 * W;
    const float *ssc = L.ssc + (size_t)seq * 128 * W;
    const RowPrep rp = row_prep(a, L, c, j);
    float4 m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 den = make_float4(0.f, 0.f, 0.f, 0.f), sum = den;
    if (active) {
        for (int q = split * (128 / NS); q < (split + 1) * (128 / NS); q++) {
            const int64_t p = 128 * (int64_t)c + q;
            float4 kv, s;
            fetch(L, skv, ssc, W, 128, p, q, j, pos0, ws_row0, kv, s);
            float *mp = &m.x, *dp_ = &den.x, *sp = &sum.x;
            const float *kp = &kv.x, *sv = &s.x;
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const float mn = fmaxf(mp[e], sv[e]);
                if (mn == -INFINITY) continue;
                const float corr = expf(mp[e] - mn);
                const float w = expf(sv[e] - mn);
                dp_[e] = dp_[e] * corr + w;
                sp[e] = sp[e] * corr + w * kp[e];
                mp[e] = mn;
            }
        }
    }
    part[0][split][t] = m;
    part[1][split][t] = den;
    part[2][split][t] = sum;
    __syncthreads();
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (split == 0 && active) {
        float *xp = &x.x;
#pragma unroll
        for (int e = 0; e < 4; e++) {
            float M = -INFINITY;
            for (int s2 = 0; s2 < NS; s2++) M = fmaxf(M, (&part[0][s2][t].x)[e]);
            float dd = 0.f, ss = 0.f;
            if (M != -INFINITY) {
                for (int s2 = 0; s2 < NS; s2++) {
                    const float ms = (&part[0][s2][t].x)[e];
                    if (ms == -INFINITY) continue;
                    const float f = expf(ms - M);
                    dd += (&part[1][s2][t].x)[e] * f;
                    ss += (&part[2][s2][t].x)[e] * f;
                }
            }
            xp[e] = dd > 0.f ? ss / dd : 0.f;
        }
    }
    // Every thread enters (the reductions use full-warp shuffles and, for
    // G > 32, block barriers); only split 0 owns the row and stores it.
    finish_row<G>(a, L, active && split == 0, seq, c, j, x, red, rp);
}

// Frontier commit (K2b): after the pools of a segment (tokens pos0 .. end-1),
// write the frontier the recurrence leaves behind.  One thread per float4
// column of W = coff*Dl, looping over the frontier rows.
__device__ __forceinline__ void commit_col(const CompressArgs &a, int lane_id, const DecodePos &dp, int decode, int seq,
                                           int col) {
    const LaneArgs L = a.lane[lane_id];
    const int ratio = a.ratio;
    const int coff = ratio == 4 ? 2 : 1;
    const int W = coff * L.Dl;
    const uint64_t pos0 = decode ? dp.pos[seq] : a.pos0;
    const uint64_t end = pos0 + (decode ? 1 : a.T);
    const int64_t ws_row0 = decode ? seq : 0;
    float *skv = L.skv + (size_t)seq * coff * ratio * W;
    float *ssc = L.ssc + (size_t)seq * coff * ratio * W;
    const uint64_t c0 = pos0 / ratio, ce = end / ratio;
    const int me = (int)(end % ratio);
    auto ws_kv = [&](uint64_t p) { return ld4(L.kv + (ws_row0 + (int64_t)(p - pos0)) * L.kv_ld + col); };
    auto ws_sc = [&](uint64_t p) {
        return add4(ld4(L.sc + (ws_row0 + (int64_t)(p - pos0)) * L.sc_ld + col), ld4(L.ape + (size_t)(p % ratio) * W + col));
    };
    if (ratio == 4) {
        // Every load first, then every store: the loads of the four row pairs go out
        // together (one memory round trip), and no store can overtake a load of the
        // frontier row it replaces.
        const bool have = ce > c0;                        // a window completed in the segment
        float4 nk[4], ns[4], mk[4], ms[4];
        bool wr4[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
            // new row q: token (ce-1)*4+q, from the segment or from the old row 4+q
            nk[q] = ns[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (have) {
                const uint64_t p = (ce - 1) * 4 + q;
                if (p >= pos0) { nk[q] = ws_kv(p); ns[q] = ws_sc(p); }
                else { nk[q] = ld4(skv + (size_t)(4 + q) * W + col); ns[q] = ld4(ssc + (size_t)(4 + q) * W + col); }
            }
            // new row 4+q: token ce*4+q of the open window when the segment reached it,
            // else (a window completed) the same token as row q
            mk[q] = nk[q]; ms[q] = ns[q];
            wr4[q] = have;
            if (q < me) {
                const uint64_t p = ce * 4 + q;
                wr4[q] = p >= pos0;
                if (wr4[q]) { mk[q] = ws_kv(p); ms[q] = ws_sc(p); }
            }
        }
#pragma unroll
        for (int q = 0; q < 4; q++) {
            if (wr4[q]) {
                st4(skv + (size_t)(4 + q) * W + col, mk[q]);
                st4(ssc + (size_t)(4 + q) * W + col, ms[q]);
            }
            if (have) {
                st4(skv + (size_t)q * W + col, nk[q]);
                st4(ssc + (size_t)q * W + col, ns[q]);
            }
        }
    } else {
        for (int q = 0; q < ratio; q++) {
            int64_t p = (q < me) ? (int64_t)(ce * ratio) + q : (int64_t)ce * ratio - ratio + q;
            if (p < 0 || (uint64_t)p < pos0) continue;
            st4(skv + (size_t)q * W + col, ws_kv((uint64_t)p));
            st4(ssc + (size_t)q * W + col, ws_sc((uint64_t)p));
        }
    }
}

__global__ void commit_kernel(CompressArgs a, int lane_id, DecodePos dp, int decode) {
    pdl_wait();
    pdl_launch_dependents();
    const LaneArgs &L = a.lane[lane_id];
    const int W = (a.ratio == 4 ? 2 : 1) * L.Dl;
    const int col = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    const int seq = decode ? blockIdx.y : 0;
    if (col >= W) return;
    if (decode && seq >= a.n_seg) return;
    commit_col(a, lane_id, dp, decode, seq, col);
}

// Decode step of a ratio-4 layer in one launch: block (sequence b, lane l)
// pools b's window when its token completes one (G = Dl/4 threads do the
// work, the rest of the block only takes part in the barriers), then, after
// the block barrier, writes the frontier the step leaves behind.
template <int GA, int GI>
__global__ void __launch_bounds__(128) compress_decode_r4_kernel(CompressArgs a, DecodePos dp) {
    __shared__ float red[32];
    // the indexer score may start now: it scores the rows of earlier steps first and waits for
    // this grid before the newest row and before finishing
    pdl_launch_dependents();
    pdl_wait();
    const int seq = blockIdx.x, lane_id = blockIdx.y;
    if (lane_id == 0) pool_r4<GA>(a, 0, dp, 1, (threadIdx.x / GA == 0) ? seq : a.n_seg, red);
    else pool_r4<GI>(a, 1, dp, 1, (threadIdx.x / GI == 0) ? seq : a.n_seg, red);
    __syncthreads();
    const int W = 2 * a.lane[lane_id].Dl;
    for (int col = threadIdx.x * 4; col < W; col += 128 * 4) commit_col(a, lane_id, dp, 1, seq, col);
}

// Prefill chunk of a ratio-4 layer in one launch for both lanes (256-thread
// blocks).  The frontier a chunk starts from is read only by the pools of the
// chunk's first two windows (c0 = pos0 / 4 takes its previous window from it,
// and both c0 and c0 + 1 take the tokens pos0 - pos0 % 4 .. pos0 - 1 from it),
// and the frontier commit rewrites it.  So block 0 pools the attention lane's
// windows c0 and c0 + 1 and then, after a block barrier, commits that lane's
// frontier; block 1 does the same for the indexer lane (windows c0 .. c0 + 7,
// eight per block); the other blocks pool the remaining windows, which read
// only the projection output.  No block waits on another.
template <int GA, int GI>
__global__ void __launch_bounds__(256) compress_prefill_r4_kernel(CompressArgs a, int att_blocks, DecodePos dp) {
    __shared__ float red[32];
    pdl_wait();
    pdl_launch_dependents();
    constexpr int PA = 256 / GA, PI = 256 / GI;          // windows per block of each lane
    const int b = blockIdx.x;
    if (b == 0 || b == 1) {
        const int lane_id = b;
        if (lane_id == 0) pool_r4<GA>(a, 0, dp, 0, threadIdx.x / GA, red);
        else pool_r4<GI>(a, 1, dp, 0, threadIdx.x / GI, red);
        __syncthreads();                                  // the frontier has been read
        const int W = 2 * a.lane[lane_id].Dl;
        for (int col = threadIdx.x * 4; col < W; col += 256 * 4) commit_col(a, lane_id, dp, 0, 0, col);
        return;
    }
    if (b < 2 + att_blocks) pool_r4<GA>(a, 0, dp, 0, PA + (b - 2) * PA + threadIdx.x / GA, red);
    else pool_r4<GI>(a, 1, dp, 0, PI + (b - 2 - att_blocks) * PI + threadIdx.x / GI, red);
}

cudaError_t pool_lane(const CompressArgs &a, int lane, const DecodePos &dp, int decode, int n_tasks, cudaStream_t s) {
    const int Dl = a.lane[lane].Dl;
    if (n_tasks <= 0) return cudaSuccess;
    if (a.ratio == 4) {
        int G = Dl / 4;
        int blocks = (n_tasks * G + 127) / 128;
        switch (G) {
            case 16: return launch_pdl(compress_r4_kernel<16>, dim3(blocks), dim3(128), 0, s, a, lane, dp, decode);
            case 32: return launch_pdl(compress_r4_kernel<32>, dim3(blocks), dim3(128), 0, s, a, lane, dp, decode);
            case 64: return launch_pdl(compress_r4_kernel<64>, dim3(blocks), dim3(128), 0, s, a, lane, dp, decode);
            case 128: return launch_pdl(compress_r4_kernel<128>, dim3(blocks), dim3(128), 0, s, a, lane, dp, decode);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (Dl / 4) {
        case 16: return launch_pdl(compress_r128_kernel<16>, dim3(n_tasks), dim3(64), 0, s, a, lane, dp, decode);
        case 32: return launch_pdl(compress_r128_kernel<32>, dim3(n_tasks), dim3(128), 0, s, a, lane, dp, decode);
        case 64: return launch_pdl(compress_r128_kernel<64>, dim3(n_tasks), dim3(256), 0, s, a, lane, dp, decode);
        case 128: return launch_pdl(compress_r128_kernel<128>, dim3(n_tasks), dim3(512), 0, s, a, lane, dp, decode);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t commit_lane(const CompressArgs &a, int lane, const DecodePos &dp, int decode, int n_seg, cudaStream_t s) {
    const int W = (a.ratio == 4 ? 2 : 1) * a.lane[lane].Dl;
    dim3 grid((W / 4 + 127) / 128, decode ? n_seg : 1);
    return launch_pdl(commit_kernel, grid, dim3(128), 0, s, a, lane, dp, decode);
}

}  // namespace

cudaError_t launch_compress_prefill(const CompressArgs &a, cudaStream_t s) {
    DecodePos dp{};
    const uint64_t n_win = (a.pos0 + a.T) / a.ratio - a.pos0 / a.ratio;
    if (a.ratio == 4 && a.n_lanes == 2) {
        const int ga = a.lane[0].Dl / 4, gi = a.lane[1].Dl / 4;
        // windows past the special blocks' first PA (attention) / PI (indexer) ones
        auto rest = [&](int per) { return n_win > (uint64_t)per ? (int)((n_win - per + per - 1) / per) : 0; };
#define DS4C_CPRE(A, I)                                                                              \
        if (ga == A && gi == I) {                                                                   \
            const int ab = rest(256 / A), ib = rest(256 / I);                                       \
            return launch_pdl(compress_prefill_r4_kernel<A, I>, dim3(2 + ab + ib), dim3(256), 0, s, a, ab, dp); \
        }
        DS4C_CPRE(128, 32)
        DS4C_CPRE(128, 16)
        DS4C_CPRE(64, 16)
        DS4C_CPRE(32, 16)
        DS4C_CPRE(128, 64)
        DS4C_CPRE(64, 32)
        DS4C_CPRE(128, 128)
        DS4C_CPRE(64, 64)
        DS4C_CPRE(32, 32)
        DS4C_CPRE(16, 16)
#undef DS4C_CPRE
    }
    for (int l = 0; l < a.n_lanes; l++) {
        cudaError_t e = pool_lane(a, l, dp, 0, (int)n_win, s);
        if (e != cudaSuccess) return e;
    }
    for (int l = 0; l < a.n_lanes; l++) {
        cudaError_t e = commit_lane(a, l, dp, 0, 1, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_compress_decode(const CompressArgs &a, const DecodePos &p, int n_seq, cudaStream_t s) {
    if (a.ratio == 4 && a.n_lanes == 2 && n_seq > 0) {
        const int ga = a.lane[0].Dl / 4, gi = a.lane[1].Dl / 4;
        const dim3 grid((unsigned)n_seq, 2);
#define DS4C_CDEC(A, I)                                                              \
        if (ga == A && gi == I) {                                                   \
            const cudaError_t e = launch_pdl(compress_decode_r4_kernel<A, I>, grid, dim3(128), 0, s, a, p); \
            if (e == cudaSuccess) pdl_prev() = PdlPrev{s, PDL_DECODE_COMPRESS};       \
            return e;                                                               \
        }
        DS4C_CDEC(128, 32)
        DS4C_CDEC(128, 16)
        DS4C_CDEC(64, 16)
        DS4C_CDEC(32, 16)
        DS4C_CDEC(128, 64)
        DS4C_CDEC(64, 32)
#undef DS4C_CDEC
    }
    for (int l = 0; l < a.n_lanes; l++) {
        cudaError_t e = pool_lane(a, l, p, 1, n_seq, s);
        if (e != cudaSuccess) return e;
    }
    for (int l = 0; l < a.n_lanes; l++) {
        cudaError_t e = commit_lane(a, l, p, 1, n_seq, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ds4c
