// extern "C" entry points of libds4c (declared in include/ds4c.h): argument
// validation on the host before any launch, workspace carving, and the launch
// sequence of each call.
#include <math.h>
#include <string.h>

#include "ds4c_internal.cuh"

using namespace ds4c;

namespace {

bool pow2_width(uint32_t w) { return w == 64 || w == 128 || w == 256 || w == 512; }
bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

namespace ds4c {

ds4c_status check_cfg(const ds4c_layer_cfg *c) {
    if (!c) return DS4C_ERR_NULL;
    if (c->ratio != 0 && c->ratio != 4 && c->ratio != 128) return DS4C_ERR_SHAPE;
    if (!pow2_width(c->head_dim)) return DS4C_ERR_SHAPE;
    if (c->d_model == 0 || c->d_model % 8) return DS4C_ERR_SHAPE;
    if (c->n_heads == 0 || c->n_heads % 8 || c->n_heads > 128) return DS4C_ERR_SHAPE;
    if ((size_t)c->n_heads * c->head_dim > 32768) return DS4C_ERR_SHAPE;
    if (c->swa == 0 || c->swa > 1024) return DS4C_ERR_SHAPE;
    if (c->dtype != DS4C_F32 && c->dtype != DS4C_BF16) return DS4C_ERR_SHAPE;
    if (c->ratio != 0) {
        if (c->n_rot < 4 || c->n_rot % 4 || c->n_rot > (uint32_t)kMaxRot || c->n_rot > c->head_dim) return DS4C_ERR_SHAPE;
        if (c->comp_cap == 0) return DS4C_ERR_SHAPE;
        if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return DS4C_ERR_SHAPE;
    }
    if (c->ratio == 4) {
        if (!pow2_width(c->idx_head_dim) || c->n_rot > c->idx_head_dim) return DS4C_ERR_SHAPE;
        if (c->top_k == 0 || c->top_k > 2048) return DS4C_ERR_SHAPE;
        if (c->idx_cap == 0 || c->idx_cap > kMaxIdxCap) return DS4C_ERR_SHAPE;
        if (c->idx_heads > 64 || c->idx_qat > 1) return DS4C_ERR_SHAPE;
        if (c->idx_qat && c->idx_head_dim != 64 && c->idx_head_dim != 128) return DS4C_ERR_SHAPE;
    }
    return DS4C_OK;
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

ds4c_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DS4C_OK;
    t_last_cuda_error = e;
    return DS4C_ERR_CUDA;
}

}  // namespace ds4c

namespace {

// Projection width of one lane (kv and score each): coff * Dl.
int proj_width(const ds4c_layer_cfg &c, bool attn) { return coff_of(c) * lane_width(c, attn); }

// Workspace layout of one call (all regions 256-byte aligned):
//   proj:   [rows][P] float, P = 2*W_attn (+ 2*W_idx on ratio-4 layers)
//           columns: attn kv | attn score | idx kv | idx score
//   scores: [rows][lds] float, lds = idx_cap rounded up to 4 (ratio 4)
//   mirror: [mirror_rows][2][head_dim] bf16 raw rows for the tensor-core
//           attention (128 + n_tok rows for a prefill chunk, 128 per sequence
//           for a decode step)
//   qsplit: the tensor-core attention's split queries, two buffers of [H][D]
//           bf16 hi + lo per CTA (one CTA per SM)
//   parts:  decode steps on the tensor-core attention split each query's rows
//           over `parts` work items: [n_seq*parts][H][D] + [n_seq*parts][2][H] float
//   gemm:   decode steps of bf16 layers with at most 128 sequences: split-K
//           partials of the projections, [kSplitK][rows][P] float
//   tail:   prefill of bf16 layers: the projection's last-round tiles split
//           along K, one 128 x 256 float partial per SM
//   qheads: ratio-4 layers with indexer heads and the round trip: the heads'
//           query vectors after it, [rows][idx_heads][idx_head_dim] float
constexpr int kSplitK = 16;
struct WsLayout {
    size_t proj_off, proj_ld;
    size_t scores_off, scores_ld;
    size_t mirror_off;
    size_t qsplit_off;
    size_t part_o_off, part_ml_off;
    size_t gemm_part_off;            // 0: no split-K region
    size_t gemm_tail_off;            // 0: no tail region
    size_t qheads_off;               // 0: no region
    int parts;
    size_t total;
};

bool tc_attention(const ds4c_layer_cfg &c) {
    return attn_tc_supported((int)c.n_heads, (int)c.head_dim, (int)c.swa, (int)c.ratio, (int)c.top_k);
}

WsLayout ws_layout(const ds4c_layer_cfg &c, uint32_t rows, uint64_t mirror_rows, bool decode) {
    WsLayout L{};
    size_t P = 0;
    if (c.ratio != 0) P = 2 * (size_t)proj_width(c, true) + (c.ratio == 4 ? 2 * (size_t)proj_width(c, false) : 0);
    L.proj_ld = P;
    L.proj_off = 0;
    size_t o = align_up(sizeof(float) * P * rows, 256);
    L.scores_ld = (c.ratio == 4) ? align_up(c.idx_cap, 4) : 0;
    L.scores_off = o;
    o += align_up(sizeof(float) * L.scores_ld * rows, 256);
    L.mirror_off = o;
    L.parts = 1;
    if (tc_attention(c)) {
        o += align_up((size_t)mirror_rows * 2 * c.head_dim * sizeof(uint16_t), 256);
        L.qsplit_off = o;
        o += align_up(attn_tc_qsplit_bytes((int)c.n_heads, (int)c.head_dim), 256);
        if (decode) {
            L.parts = attn_tc_decode_parts((int)c.ratio, (int)c.top_k, (int)c.comp_cap);
            const size_t items = (size_t)rows * L.parts;
            L.part_o_off = o;
            o += align_up(items * c.n_heads * c.head_dim * sizeof(float), 256);
            L.part_ml_off = o;
            o += align_up(items * 2 * c.n_heads * sizeof(float), 256);
        }
    }
    if (decode && c.dtype == DS4C_BF16 && P > 0 && rows <= 128) {
        L.gemm_part_off = o;
        o += align_up(sizeof(float) * (size_t)kSplitK * rows * P, 256);
    }
    if (!decode && c.dtype == DS4C_BF16 && P > 0) {
        L.gemm_tail_off = o;
        o += align_up(sizeof(float) * gemm_tail_floats(), 256);
    }
    if (c.ratio == 4 && c.idx_heads > 0 && c.idx_qat) {
        L.qheads_off = o;
        o += align_up(sizeof(float) * (size_t)rows * c.idx_heads * c.idx_head_dim, 256);
    }
    L.total = o < 256 ? 256 : o;
    return L;
}
WsLayout ws_prefill(const ds4c_layer_cfg &c, uint32_t n_tok) { return ws_layout(c, n_tok, 128 + (uint64_t)n_tok, false); }
WsLayout ws_decode(const ds4c_layer_cfg &c, uint32_t n_seq) { return ws_layout(c, n_seq, 128 * (uint64_t)n_seq, true); }

RopeTable rope_table(const ds4c_layer_cfg &c) {
    RopeTable t;
    memset(&t, 0, sizeof t);
    for (uint32_t i = 0; i < c.n_rot / 2; i++)
        t.inv_freq[i] = (float)pow((double)c.rope_base, -2.0 * (double)i / (double)c.n_rot);
    return t;
}

ds4c_status check_lane_state(const ds4c_lane_state &s) {
    if (!s.comp || !s.state_kv || !s.state_score) return DS4C_ERR_NULL;
    if (!aligned16(s.comp) || !aligned16(s.state_kv) || !aligned16(s.state_score) || !aligned16(s.prequant))
        return DS4C_ERR_SHAPE;
    return DS4C_OK;
}

ds4c_status check_lane_weights(const ds4c_lane_weights *w) {
    if (!w || !w->wkv || !w->wgate || !w->ape) return DS4C_ERR_NULL;
    if (!aligned16(w->wkv) || !aligned16(w->wgate) || !aligned16(w->ape) || !aligned16(w->norm)) return DS4C_ERR_SHAPE;
    return DS4C_OK;
}

// Shared front half of prefill and decode compression: projections into the
// workspace, then the fused compressor.
ds4c_status run_compress(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *aw, const ds4c_lane_weights *iw,
                         const ds4c_layer_state *st, const void *hidden, uint32_t rows, uint64_t pos0,
                         const DecodePos *dp, void *ws, cudaStream_t stream, cudaEvent_t after_projection = nullptr) {
    const ds4c_layer_cfg &c = *cfg;
    const WsLayout L = (dp == nullptr) ? ws_prefill(c, rows) : ws_decode(c, rows);
    float *proj = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.proj_off);
    const int Wa = proj_width(c, true), Wi = proj_width(c, false);
    GemmArgs g{};
    g.A = hidden;
    g.M = (int)rows;
    g.K = (int)c.d_model;
    g.dtype = (int)c.dtype;
    g.n_groups = 2;
    g.g[0] = GemmGroup{aw->wkv, proj, (int64_t)L.proj_ld, Wa};
    g.g[1] = GemmGroup{aw->wgate, proj + Wa, (int64_t)L.proj_ld, Wa};
    if (c.ratio == 4) {
        g.n_groups = 4;
        g.g[2] = GemmGroup{iw->wkv, proj + 2 * Wa, (int64_t)L.proj_ld, Wi};
        g.g[3] = GemmGroup{iw->wgate, proj + 2 * Wa + Wi, (int64_t)L.proj_ld, Wi};
    }
    if (L.gemm_part_off != 0) {
        g.c_base = proj;
        g.part = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.gemm_part_off);
        g.part_ld = (int64_t)L.proj_ld;
        g.max_ksplit = kSplitK;
    }
    if (L.gemm_tail_off != 0) g.tail_buf = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.gemm_tail_off);
    cudaError_t e = cudaErrorNotSupported;
    if (c.dtype == DS4C_BF16) e = launch_gemm_tc(g, stream);
    if (e == cudaErrorNotSupported) e = launch_gemm_simt(g, stream);
    if (e != cudaSuccess) return cuda_status(e);
    if (after_projection && (e = cudaEventRecord(after_projection, stream)) != cudaSuccess) return cuda_status(e);

    CompressArgs a{};
    a.n_lanes = (c.ratio == 4) ? 2 : 1;
    a.ratio = (int)c.ratio;
    a.n_rot = (int)c.n_rot;
    a.eps = c.rms_eps;
    a.rope = rope_table(c);
    for (int l = 0; l < a.n_lanes; l++) {
        const bool attn = l == 0;
        const ds4c_lane_weights *w = attn ? aw : iw;
        const ds4c_lane_state &s = attn ? st->attn : st->idx;
        LaneArgs &la = a.lane[l];
        const int col0 = attn ? 0 : 2 * Wa;
        const int W = attn ? Wa : Wi;
        la.kv = proj + col0;
        la.kv_ld = (int64_t)L.proj_ld;
        la.sc = proj + col0 + W;
        la.sc_ld = (int64_t)L.proj_ld;
        la.ape = w->ape;
        la.gain = w->norm;
        la.comp = s.comp;
        la.prequant = s.prequant;
        la.skv = s.state_kv;
        la.ssc = s.state_score;
        la.split = (attn && tc_attention(c)) ? s.comp_split : nullptr;
        la.Dl = lane_width(c, attn);
        la.cap = (int)(attn ? c.comp_cap : c.idx_cap);
        la.is_attn = attn ? 1 : 0;
        la.qat = (!attn && c.idx_qat) ? 1 : 0;
        la.qat_c = (float)(1.0 / sqrt((double)la.Dl));
    }
    if (dp == nullptr) {
        a.n_seg = 1;
        a.pos0 = pos0;
        a.T = rows;
        e = launch_compress_prefill(a, stream);
    } else {
        a.n_seg = (int)rows;
        e = launch_compress_decode(a, *dp, (int)rows, stream);
    }
    return cuda_status(e);
}

// Per-sequence strides of the state arrays.
size_t raw_stride(const ds4c_layer_cfg &c) { return (size_t)c.swa * c.head_dim; }
size_t comp_stride(const ds4c_layer_cfg &c, bool attn) {
    return (size_t)(attn ? c.comp_cap : c.idx_cap) * lane_width(c, attn);
}
size_t frontier_stride(const ds4c_layer_cfg &c, bool attn) {
    const int coff = coff_of(c);
    const int rows = attn ? coff * (int)c.ratio : 8;
    return (size_t)rows * (attn ? coff : 2) * lane_width(c, attn);
}

}  // namespace

extern "C" {

const char *ds4c_status_string(ds4c_status s) {
    switch (s) {
        case DS4C_OK: return "ok";
        case DS4C_ERR_NULL: return "a required pointer is NULL";
        case DS4C_ERR_SHAPE: return "configuration, size or alignment outside the supported set";
        case DS4C_ERR_CAPACITY: return "positions beyond the state capacity, or output buffer too small";
        case DS4C_ERR_UNSUPPORTED: return "unsupported call form (n_seq > 1 with n_tok > 1, or batch too large)";
        case DS4C_ERR_CUDA: return "CUDA runtime error";
        case DS4C_ERR_DEVICE: return "a kernel reported a device-side failure";
        case DS4C_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

size_t ds4c_workspace_bytes(const ds4c_layer_cfg *cfg, uint32_t max_tok, uint32_t max_seq) {
    if (check_cfg(cfg) != DS4C_OK) return 0;
    const size_t a = ws_prefill(*cfg, max_tok > 0 ? max_tok : 1).total;
    const size_t b = max_seq > 0 ? ws_decode(*cfg, max_seq).total : 0;
    return a > b ? a : b;
}

ds4c_status ds4c_fma_probe(uint32_t blocks, uint32_t iters, float *out, double *flops_h, cudaStream_t stream) {
    if (!out || !flops_h) return DS4C_ERR_NULL;
    if (blocks == 0 || iters == 0 || iters > (1u << 24)) return DS4C_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0) return DS4C_ERR_SHAPE;
    *flops_h = fma_probe_flops(blocks, iters);
    return cuda_status(launch_fma_probe(blocks, iters, out, stream));
}

int ds4c_attn_uses_tensor_cores(const ds4c_layer_cfg *cfg) {
    if (check_cfg(cfg) != DS4C_OK) return 0;
    return tc_attention(*cfg) ? 1 : 0;
}

ds4c_status ds4c_state_init(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st, uint32_t n_seq, cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    if (!st || !st->raw) return DS4C_ERR_NULL;
    if (n_seq == 0) return DS4C_ERR_SHAPE;
    const ds4c_layer_cfg &c = *cfg;
    if (c.ratio != 0 && (s = check_lane_state(st->attn)) != DS4C_OK) return s;
    if (c.ratio == 4 && (s = check_lane_state(st->idx)) != DS4C_OK) return s;
    cudaError_t e = launch_fill(st->raw, raw_stride(c) * n_seq, 0.f, stream);
    if (e == cudaSuccess && c.ratio != 0) {
        e = launch_fill(st->attn.state_kv, frontier_stride(c, true) * n_seq, 0.f, stream);
        if (e == cudaSuccess) e = launch_fill(st->attn.state_score, frontier_stride(c, true) * n_seq, -INFINITY, stream);
    }
    if (e == cudaSuccess && c.ratio == 4) {
        e = launch_fill(st->idx.state_kv, frontier_stride(c, false) * n_seq, 0.f, stream);
        if (e == cudaSuccess) e = launch_fill(st->idx.state_score, frontier_stride(c, false) * n_seq, -INFINITY, stream);
    }
    return cuda_status(e);
}

static ds4c_status compress_prefill_impl(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                         const ds4c_lane_weights *idx, const ds4c_layer_state *st,
                                         const void *hidden, uint32_t n_tok, uint64_t pos0, void *ws,
                                         size_t ws_bytes, cudaStream_t stream, cudaEvent_t after_projection) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (c.ratio == 0 || n_tok == 0) return DS4C_OK;
    if (!st || !hidden) return DS4C_ERR_NULL;
    if ((s = check_lane_weights(attn)) != DS4C_OK) return s;
    if ((s = check_lane_state(st->attn)) != DS4C_OK) return s;
    if (c.ratio == 4) {
        if ((s = check_lane_weights(idx)) != DS4C_OK) return s;
        if ((s = check_lane_state(st->idx)) != DS4C_OK) return s;
    } else if (idx != nullptr) {
        return DS4C_ERR_SHAPE;
    }
    if (!aligned16(hidden)) return DS4C_ERR_SHAPE;
    const uint64_t end = pos0 + n_tok;
    if (end / c.ratio > c.comp_cap) return DS4C_ERR_CAPACITY;
    if (c.ratio == 4 && end / 4 > c.idx_cap) return DS4C_ERR_CAPACITY;
    if (tc_attention(c) && !st->attn.comp_split) return DS4C_ERR_NULL;
    if (!ws) return DS4C_ERR_WORKSPACE;
    if (ws_bytes < ws_prefill(c, n_tok).total) return DS4C_ERR_WORKSPACE;
    return run_compress(cfg, attn, idx, st, hidden, n_tok, pos0, nullptr, ws, stream, after_projection);
}

ds4c_status ds4c_compress_prefill(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                  const ds4c_lane_weights *idx, const ds4c_layer_state *st,
                                  const void *hidden, uint32_t n_tok, uint64_t pos0,
                                  void *ws, size_t ws_bytes, cudaStream_t stream) {
    return compress_prefill_impl(cfg, attn, idx, st, hidden, n_tok, pos0, ws, ws_bytes, stream, nullptr);
}

ds4c_status ds4c_compress_prefill_timed(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                        const ds4c_lane_weights *idx, const ds4c_layer_state *st,
                                        const void *hidden, uint32_t n_tok, uint64_t pos0, void *ws,
                                        size_t ws_bytes, cudaEvent_t after_projection, cudaStream_t stream) {
    if (!after_projection) return DS4C_ERR_NULL;
    return compress_prefill_impl(cfg, attn, idx, st, hidden, n_tok, pos0, ws, ws_bytes, stream, after_projection);
}

ds4c_status ds4c_compress_decode_step(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                      const ds4c_lane_weights *idx, const ds4c_layer_state *st,
                                      const void *hidden, const uint64_t *pos_h, uint32_t n_seq,
                                      void *ws, size_t ws_bytes, cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (n_seq == 0) return DS4C_ERR_SHAPE;
    if (n_seq > (uint32_t)kMaxDecodeSeq) return DS4C_ERR_UNSUPPORTED;
    if (!pos_h) return DS4C_ERR_NULL;
    if (c.ratio == 0) return DS4C_OK;
    if (!st || !hidden) return DS4C_ERR_NULL;
    if ((s = check_lane_weights(attn)) != DS4C_OK) return s;
    if ((s = check_lane_state(st->attn)) != DS4C_OK) return s;
    if (c.ratio == 4) {
        if ((s = check_lane_weights(idx)) != DS4C_OK) return s;
        if ((s = check_lane_state(st->idx)) != DS4C_OK) return s;
    } else if (idx != nullptr) {
        return DS4C_ERR_SHAPE;
    }
    if (!aligned16(hidden)) return DS4C_ERR_SHAPE;
    DecodePos dp;
    for (uint32_t b = 0; b < n_seq; b++) {
        const uint64_t end = pos_h[b] + 1;
        if (end / c.ratio > c.comp_cap) return DS4C_ERR_CAPACITY;
        if (c.ratio == 4 && end / 4 > c.idx_cap) return DS4C_ERR_CAPACITY;
        dp.pos[b] = pos_h[b];
    }
    if (tc_attention(c) && !st->attn.comp_split) return DS4C_ERR_NULL;
    if (!ws) return DS4C_ERR_WORKSPACE;
    if (ws_bytes < ws_decode(c, n_seq).total) return DS4C_ERR_WORKSPACE;
    return run_compress(cfg, attn, idx, st, hidden, n_seq, 0, &dp, ws, stream);
}

ds4c_status ds4c_indexer_topk(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st, const float *q_idx,
                              const uint64_t *pos_h, uint32_t n_seq, uint32_t n_tok, int32_t *topk,
                              float *scores, size_t score_stride, void *ws, size_t ws_bytes, cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (c.ratio != 4) return DS4C_ERR_SHAPE;
    if (n_seq == 0 || n_tok == 0) return DS4C_ERR_SHAPE;
    if (n_seq > 1 && n_tok > 1) return DS4C_ERR_UNSUPPORTED;
    if (n_seq > (uint32_t)kMaxDecodeSeq) return DS4C_ERR_UNSUPPORTED;
    if (!st || !q_idx || !pos_h || !topk) return DS4C_ERR_NULL;
    if (!st->idx.comp) return DS4C_ERR_NULL;
    if (!aligned16(q_idx) || !aligned16(st->idx.comp) || !aligned16(topk) || !aligned16(scores)) return DS4C_ERR_SHAPE;
    const uint32_t rows = n_seq * n_tok;
    uint64_t vis_max = 0;
    DecodePos dp;
    if (n_seq == 1) {
        vis_max = (pos_h[0] + n_tok) / 4;
    } else {
        for (uint32_t b = 0; b < n_seq; b++) {
            dp.pos[b] = pos_h[b];
            const uint64_t v = (pos_h[b] + 1) / 4;
            vis_max = v > vis_max ? v : vis_max;
        }
    }
    if (vis_max > c.idx_cap) return DS4C_ERR_CAPACITY;
    if (scores && score_stride < vis_max) return DS4C_ERR_CAPACITY;
    if (!ws) return DS4C_ERR_WORKSPACE;
    const WsLayout L = (n_seq == 1) ? ws_prefill(c, rows) : ws_decode(c, rows);
    if (ws_bytes < L.total) return DS4C_ERR_WORKSPACE;
    IndexerArgs a{};
    a.q = q_idx;
    a.rows = st->idx.comp;
    a.seq_stride = (int64_t)c.idx_cap * c.idx_head_dim;
    if (scores) {
        a.scores = scores;
        a.lds = (int64_t)score_stride;
    } else {
        a.scores = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.scores_off);
        a.lds = (int64_t)L.scores_ld;
    }
    a.topk = topk;
    a.d = (int)c.idx_head_dim;
    a.k = (int)c.top_k;
    a.n_seq = (int)n_seq;
    a.n_tok = (int)n_tok;
    a.pos0 = pos_h[0];
    cudaError_t e = (n_seq == 1) ? launch_indexer_prefill(a, stream) : launch_indexer_decode(a, dp, stream);
    return cuda_status(e);
}

ds4c_status ds4c_indexer_topk_heads(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st, const float *q_idx,
                                    const float *w_idx, const uint64_t *pos_h, uint32_t n_seq, uint32_t n_tok,
                                    int32_t *topk, float *scores, size_t score_stride, void *ws, size_t ws_bytes,
                                    cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (c.ratio != 4 || c.idx_heads == 0) return DS4C_ERR_SHAPE;
    if (c.idx_head_dim != 64 && c.idx_head_dim != 128) return DS4C_ERR_SHAPE;
    if (n_seq == 0 || n_tok == 0) return DS4C_ERR_SHAPE;
    if (n_seq > 1 && n_tok > 1) return DS4C_ERR_UNSUPPORTED;
    if (n_seq > (uint32_t)kMaxDecodeSeq) return DS4C_ERR_UNSUPPORTED;
    if (!st || !q_idx || !w_idx || !pos_h || !topk || !st->idx.comp) return DS4C_ERR_NULL;
    if (!aligned16(q_idx) || !aligned16(w_idx) || !aligned16(st->idx.comp) || !aligned16(topk) || !aligned16(scores))
        return DS4C_ERR_SHAPE;
    const uint32_t rows = n_seq * n_tok;
    uint64_t vis_max = 0;
    DecodePos dp;
    if (n_seq == 1) {
        vis_max = (pos_h[0] + n_tok) / 4;
    } else {
        for (uint32_t b = 0; b < n_seq; b++) {
            dp.pos[b] = pos_h[b];
            const uint64_t v = (pos_h[b] + 1) / 4;
            vis_max = v > vis_max ? v : vis_max;
        }
    }
    if (vis_max > c.idx_cap) return DS4C_ERR_CAPACITY;
    if (scores && score_stride < vis_max) return DS4C_ERR_CAPACITY;
    if (!ws) return DS4C_ERR_WORKSPACE;
    const WsLayout L = (n_seq == 1) ? ws_prefill(c, rows) : ws_decode(c, rows);
    if (ws_bytes < L.total) return DS4C_ERR_WORKSPACE;
    IndexerArgs a{};
    a.q = q_idx;
    if (c.idx_qat) {
        // the heads' query vectors take the same round trip as the rows
        float *qh = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.qheads_off);
        cudaError_t e = launch_qat_vectors(q_idx, qh, (int64_t)rows * c.idx_heads, (int)c.idx_head_dim,
                                           (float)(1.0 / sqrt((double)c.idx_head_dim)), stream);
        if (e != cudaSuccess) return cuda_status(e);
        a.q = qh;
    }
    a.rows = st->idx.comp;
    a.seq_stride = (int64_t)c.idx_cap * c.idx_head_dim;
    if (scores) {
        a.scores = scores;
        a.lds = (int64_t)score_stride;
    } else {
        a.scores = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.scores_off);
        a.lds = (int64_t)L.scores_ld;
    }
    a.topk = topk;
    a.d = (int)c.idx_head_dim;
    a.k = (int)c.top_k;
    a.n_seq = (int)n_seq;
    a.n_tok = (int)n_tok;
    a.pos0 = pos_h[0];
    return cuda_status(launch_indexer_heads(a, w_idx, (int)c.idx_heads, n_seq > 1 ? &dp : nullptr, stream));
}

ds4c_status ds4c_sparse_swa_attn(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st, const float *q,
                                 const float *raw_new, const int32_t *topk, const uint64_t *pos_h,
                                 uint32_t n_seq, uint32_t n_tok, float *out, int commit_ring, void *ws,
                                 size_t ws_bytes, cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (n_seq == 0 || n_tok == 0) return DS4C_ERR_SHAPE;
    if (n_seq > 1 && n_tok > 1) return DS4C_ERR_UNSUPPORTED;
    if (n_seq > (uint32_t)kMaxDecodeSeq) return DS4C_ERR_UNSUPPORTED;
    if (!st || !st->raw || !q || !raw_new || !pos_h || !out) return DS4C_ERR_NULL;
    if (c.ratio != 0 && !st->attn.comp) return DS4C_ERR_NULL;
    if (c.ratio == 4 && !topk) return DS4C_ERR_NULL;
    if (!aligned16(q) || !aligned16(raw_new) || !aligned16(out) || !aligned16(st->raw) || !aligned16(st->attn.comp) ||
        !aligned16(topk))
        return DS4C_ERR_SHAPE;
    DecodePos dp;
    if (n_seq == 1) {
        const uint64_t end = pos_h[0] + n_tok;
        if (c.ratio != 0 && end / c.ratio > c.comp_cap) return DS4C_ERR_CAPACITY;
    } else {
        for (uint32_t b = 0; b < n_seq; b++) {
            dp.pos[b] = pos_h[b];
            if (c.ratio != 0 && (pos_h[b] + 1) / c.ratio > c.comp_cap) return DS4C_ERR_CAPACITY;
        }
    }
    cudaError_t e;
    bool ring_done = false;   // the decode combine wrote the ring slots
    if (tc_attention(c)) {
        if (c.ratio != 0 && !st->attn.comp_split) return DS4C_ERR_NULL;
        const WsLayout L = (n_seq == 1) ? ws_prefill(c, n_tok) : ws_decode(c, n_seq);
        if (!ws) return DS4C_ERR_WORKSPACE;
        if (ws_bytes < L.total) return DS4C_ERR_WORKSPACE;
        AttnTcArgs a{};
        a.q = q;
        a.raw_new = raw_new;
        a.ring = st->raw;
        a.comp_split = st->attn.comp_split;
        a.raw_mirror = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(ws) + L.mirror_off);
        a.qsplit = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(ws) + L.qsplit_off);
        a.topk = topk;
        a.out = out;
        a.D = (int)c.head_dim;
        a.H = (int)c.n_heads;
        a.ratio = (int)c.ratio;
        a.k = (int)c.top_k;
        a.comp_cap = (int)c.comp_cap;
        a.n_rot = (int)c.n_rot;
        a.S = (int)c.swa;
        a.scale = c.attn_scale;
        a.n_seq = (int)n_seq;
        a.n_tok = (int)n_tok;
        a.n_seq_state = (int)n_seq;
        a.pos0 = pos_h[0];
        a.parts = (n_seq > 1) ? L.parts : 1;
        a.part_o = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.part_o_off);
        a.part_ml = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.part_ml_off);
        a.commit_ring = (commit_ring && a.parts > 1) ? 1 : 0;
        ring_done = a.commit_ring != 0;
        e = launch_attention_tc(a, n_seq > 1 ? &dp : nullptr, stream);
    } else {
        AttnArgs a{};
        a.q = q;
        a.raw_new = raw_new;
        a.ring = st->raw;
        a.comp = st->attn.comp;
        a.topk = topk;
        a.out = out;
        a.D = (int)c.head_dim;
        a.H = (int)c.n_heads;
        a.S = (int)c.swa;
        a.ratio = (int)c.ratio;
        a.k = (int)c.top_k;
        a.comp_cap = (int)c.comp_cap;
        a.scale = c.attn_scale;
        a.n_seq = (int)n_seq;
        a.n_tok = (int)n_tok;
        a.pos0 = pos_h[0];
        e = launch_attention(a, n_seq > 1 ? &dp : nullptr, stream);
    }
    if (e == cudaSuccess && commit_ring && !ring_done)
        e = launch_ring_commit(st->raw, raw_new, (int)c.head_dim, (int)c.swa, (int)n_seq, (int)n_tok, pos_h[0],
                               n_seq > 1 ? &dp : nullptr, stream);
    return cuda_status(e);
}

size_t ds4c_checkpoint_floats(const ds4c_layer_cfg *cfg, uint64_t pos) {
    if (check_cfg(cfg) != DS4C_OK) return 0;
    const ds4c_layer_cfg &c = *cfg;
    const uint64_t n_live = pos < c.swa ? pos : c.swa;
    size_t total = (size_t)n_live * c.head_dim;
    if (c.ratio != 0) total += (size_t)(pos / c.ratio) * c.head_dim + 2 * frontier_stride(c, true);
    if (c.ratio == 4) total += (size_t)(pos / 4) * c.idx_head_dim + 2 * frontier_stride(c, false);
    return total;
}

ds4c_status ds4c_checkpoint_gather(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st, uint32_t seq,
                                   uint64_t pos, float *dst, size_t dst_floats, size_t *written_h,
                                   cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (!st || !st->raw || !dst) return DS4C_ERR_NULL;
    if (c.ratio != 0 && (s = check_lane_state(st->attn)) != DS4C_OK) return s;
    if (c.ratio == 4 && (s = check_lane_state(st->idx)) != DS4C_OK) return s;
    if (c.ratio != 0 && pos / c.ratio > c.comp_cap) return DS4C_ERR_CAPACITY;
    if (c.ratio == 4 && pos / 4 > c.idx_cap) return DS4C_ERR_CAPACITY;
    const size_t need = ds4c_checkpoint_floats(cfg, pos);
    if (dst_floats < need) return DS4C_ERR_CAPACITY;
    GatherArgs a{};
    a.dst = dst;
    a.ring = st->raw + (size_t)seq * raw_stride(c);
    a.D = c.head_dim;
    a.S = c.swa;
    a.pos = pos;
    a.n_live = (int64_t)(pos < c.swa ? pos : c.swa);
    int64_t o = a.n_live * a.D;
    int n = 0;
    if (c.ratio != 0) {
        const size_t fs = frontier_stride(c, true);
        a.seg[n++] = GatherSeg{st->attn.comp + (size_t)seq * comp_stride(c, true), o, (int64_t)(pos / c.ratio) * c.head_dim};
        o += a.seg[n - 1].n;
        a.seg[n++] = GatherSeg{st->attn.state_kv + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
        a.seg[n++] = GatherSeg{st->attn.state_score + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
    }
    if (c.ratio == 4) {
        const size_t fs = frontier_stride(c, false);
        a.seg[n++] = GatherSeg{st->idx.comp + (size_t)seq * comp_stride(c, false), o, (int64_t)(pos / 4) * c.idx_head_dim};
        o += a.seg[n - 1].n;
        a.seg[n++] = GatherSeg{st->idx.state_kv + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
        a.seg[n++] = GatherSeg{st->idx.state_score + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
    }
    a.n_seg = n;
    if ((size_t)o != need) return DS4C_ERR_SHAPE;
    if (written_h) *written_h = need;
    return cuda_status(launch_gather(a, stream));
}

ds4c_status ds4c_checkpoint_scatter(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st, uint32_t seq,
                                    uint64_t pos, const float *src, size_t src_floats, cudaStream_t stream) {
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (!st || !st->raw || !src) return DS4C_ERR_NULL;
    if (c.ratio != 0 && (s = check_lane_state(st->attn)) != DS4C_OK) return s;
    if (c.ratio == 4 && (s = check_lane_state(st->idx)) != DS4C_OK) return s;
    if (c.ratio != 0 && tc_attention(c) && !st->attn.comp_split) return DS4C_ERR_NULL;
    if (c.ratio != 0 && pos / c.ratio > c.comp_cap) return DS4C_ERR_CAPACITY;
    if (c.ratio == 4 && pos / 4 > c.idx_cap) return DS4C_ERR_CAPACITY;
    const size_t need = ds4c_checkpoint_floats(cfg, pos);
    if (src_floats < need) return DS4C_ERR_CAPACITY;
    ScatterArgs a{};
    a.src = src;
    a.ring = st->raw + (size_t)seq * raw_stride(c);
    a.D = c.head_dim;
    a.S = c.swa;
    a.pos = pos;
    a.n_live = (int64_t)(pos < c.swa ? pos : c.swa);
    int64_t o = a.n_live * a.D;
    int n = 0;
    float *comp_attn = nullptr;
    int64_t n_comp = 0;
    if (c.ratio != 0) {
        const size_t fs = frontier_stride(c, true);
        comp_attn = st->attn.comp + (size_t)seq * comp_stride(c, true);
        n_comp = (int64_t)(pos / c.ratio);
        a.seg[n++] = ScatterSeg{comp_attn, o, n_comp * c.head_dim};
        o += a.seg[n - 1].n;
        a.seg[n++] = ScatterSeg{st->attn.state_kv + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
        a.seg[n++] = ScatterSeg{st->attn.state_score + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
    }
    if (c.ratio == 4) {
        const size_t fs = frontier_stride(c, false);
        a.seg[n++] = ScatterSeg{st->idx.comp + (size_t)seq * comp_stride(c, false), o, (int64_t)(pos / 4) * c.idx_head_dim};
        o += a.seg[n - 1].n;
        a.seg[n++] = ScatterSeg{st->idx.state_kv + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
        a.seg[n++] = ScatterSeg{st->idx.state_score + (size_t)seq * fs, o, (int64_t)fs};
        o += (int64_t)fs;
    }
    a.n_seg = n;
    if ((size_t)o != need) return DS4C_ERR_SHAPE;
    cudaError_t e = launch_scatter(a, stream);
    // the tensor-core attention's bf16 mirror of the restored compressed rows
    if (e == cudaSuccess && c.ratio != 0 && tc_attention(c))
        e = launch_split_rows(st->attn.comp_split + (size_t)seq * c.comp_cap * 2 * c.head_dim, comp_attn, n_comp,
                              (int)c.head_dim, stream);
    return cuda_status(e);
}

ds4c_status ds4c_payload_header(const ds4c_payload_info *info, uint32_t out[DS4C_PAYLOAD_U32_FIELDS]) {
    if (!info || !out) return DS4C_ERR_NULL;
    const uint32_t f[DS4C_PAYLOAD_U32_FIELDS] = {DS4C_PAYLOAD_MAGIC,        DS4C_PAYLOAD_VERSION,   info->ctx_size,
                                                 info->prefill_chunk,      info->raw_cap,          info->raw_window,
                                                 info->comp_cap,           info->token_count,      info->layer_count,
                                                 info->head_dim,           info->idx_head_dim,     info->vocab_size,
                                                 info->live_raw_rows};
    for (unsigned i = 0; i < DS4C_PAYLOAD_U32_FIELDS; i++) out[i] = f[i];
    return DS4C_OK;
}

const char *ds4c_last_cuda_error(void) { return cudaGetErrorName(t_last_cuda_error); }

ds4c_status ds4c_test_set_wait_limit(uint64_t limit_ns) {
    const unsigned long long ns = limit_ns ? limit_ns : kWaitNsDefault;
    cudaError_t e = gemm_tc_set_wait_ns(ns);
    if (e == cudaSuccess) e = attn_tc_set_wait_ns(ns);
    if (e == cudaSuccess) e = idx_set_wait_ns(ns);
    return cuda_status(e);
}

ds4c_status ds4c_test_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
    return cuda_status(launch_wait_selftest(limit_ns, stream));
}

ds4c_status ds4c_sync_status(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_status(e);
    const unsigned int e1 = gemm_tc_read_clear_error(), e2 = attn_tc_read_clear_error(), e3 = idx_read_clear_error();
    if (e1 != 0 || e2 != 0 || e3 != 0) return DS4C_ERR_DEVICE;
    return DS4C_OK;
}

}  // extern "C"
