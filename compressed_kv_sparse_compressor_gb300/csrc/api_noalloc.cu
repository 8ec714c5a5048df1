// ds4c_indexer_topk_noalloc: the indexer top-k call for callers that cannot
// allocate device memory.
//
// Some callers have no way to allocate: a runtime that owns every byte of
// device memory through its own pool and forbids cudaMalloc on the serving
// path (allocation may synchronise the device or fragment the pool), code that
// runs inside a framework hook without access to an allocator, or a caller
// that must not stall on the allocator at all.  They cannot hand over the
// workspace ds4c_indexer_topk needs for its score matrix.  This entry point
// keeps that score matrix in a fixed file-scope device array instead, so the
// caller passes only its inputs and outputs.
//
// The array is DS4C_NOALLOC_SCORE_FLOATS floats (8 MiB).  Every GPU that loads
// the library holds it until the process exits, and every call shares it:
// two calls whose kernels overlap on the GPU (different streams without
// ordering between them) race on it.  A call only reads score entries that the
// same call wrote first, so nothing in the array has to start at zero.
#include <mutex>

#include "ds4c_internal.cuh"

using namespace ds4c;

namespace {

static __device__ __align__(256) float g_noalloc_scores[DS4C_NOALLOC_SCORE_FLOATS];

constexpr int kMaxDevices = 64;
float *g_scores_dev[kMaxDevices] = {};
std::mutex g_scores_mu;

// Device address of the array on the current device.  The first call on each
// device looks it up with that device current; later calls reuse it.  The
// cached address belongs to the CUDA context of that first call: after a
// cudaDeviceReset of that device the module is loaded anew and the address
// is stale, so this entry point must not be used across a device reset.
cudaError_t scores_on_current_device(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scores_mu);
    if (!g_scores_dev[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scores);
        if (e != cudaSuccess) return e;
        g_scores_dev[dev] = static_cast<float *>(p);
    }
    *out = g_scores_dev[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15) == 0; }

}  // namespace

extern "C" ds4c_status ds4c_indexer_topk_noalloc(const ds4c_layer_cfg *cfg, const ds4c_layer_state *st,
                                                 const float *q_idx, const uint64_t *pos_h, uint32_t n_seq,
                                                 uint32_t n_tok, int32_t *topk, cudaStream_t stream) {
    // the same shape rules as ds4c_indexer_topk
    ds4c_status s = check_cfg(cfg);
    if (s != DS4C_OK) return s;
    const ds4c_layer_cfg &c = *cfg;
    if (c.ratio != 4) return DS4C_ERR_SHAPE;
    if (n_seq == 0 || n_tok == 0) return DS4C_ERR_SHAPE;
    if (n_seq > 1 && n_tok > 1) return DS4C_ERR_UNSUPPORTED;
    if (n_seq > (uint32_t)kMaxDecodeSeq) return DS4C_ERR_UNSUPPORTED;
    if (!st || !q_idx || !pos_h || !topk || !st->idx.comp) return DS4C_ERR_NULL;
    if (!aligned16(q_idx) || !aligned16(st->idx.comp) || !aligned16(topk)) return DS4C_ERR_SHAPE;
    uint64_t vis_max = 0;
    DecodePos dp{};
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
    // the score matrix [n_seq * n_tok][lds] must fit the fixed array
    const uint64_t lds = (vis_max + 3) / 4 * 4;
    const uint64_t rows = (uint64_t)n_seq * n_tok;
    if (rows * (lds > 0 ? lds : 4) > (uint64_t)DS4C_NOALLOC_SCORE_FLOATS) return DS4C_ERR_CAPACITY;
    float *scores = nullptr;
    cudaError_t e = scores_on_current_device(&scores);
    if (e != cudaSuccess) return cuda_status(e);
    IndexerArgs a{};
    a.q = q_idx;
    a.rows = st->idx.comp;
    a.seq_stride = (int64_t)c.idx_cap * c.idx_head_dim;
    a.scores = scores;
    a.lds = (int64_t)(lds > 0 ? lds : 4);
    a.topk = topk;
    a.d = (int)c.idx_head_dim;
    a.k = (int)c.top_k;
    a.n_seq = (int)n_seq;
    a.n_tok = (int)n_tok;
    a.pos0 = pos_h[0];
    e = (n_seq == 1) ? launch_indexer_prefill(a, stream) : launch_indexer_decode(a, dp, stream);
    return cuda_status(e);
}
