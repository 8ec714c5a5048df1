/*
 * ds4c — compressed-KV sparse attention path of a DeepSeek-V4-style engine,
 * as hand-written CUDA for sm_103a (GB300), behind a plain C ABI.
 *
 * The method is the one described in "Metal グラフと圧縮 KV の実装を読む"
 * (DwarfStar/ds4 series part 3; cited below as [P2] with its section) and the
 * checkpoint layout of "【#4】ds4.c を読み解く" ([P1]).  Per layer and token a
 * learned compressor projects the hidden state (wkv, wgate), adds a learned
 * position bias (APE) to the score, stores both into a recurrent frontier and,
 * at every ratio boundary, softmax-pools the frontier into one row that goes
 * through RMSNorm, a RoPE on its last n_rot dims and (attention lane) an FP8
 * E4M3 round trip before it is appended to the compressed KV.  Ratio-4 layers
 * run a second (indexer) lane; a top-k over the indexer rows selects which
 * compressed rows the attention sees next to a raw sliding window (swa rows,
 * 128 in the pages' model).
 *
 * Conventions shared by every call
 *   - Tensor pointers are DEVICE pointers owned by the caller, unless a name
 *     ends in _h (host pointer).  The library allocates no device memory; its
 *     scratch is the caller's workspace, sized by ds4c_workspace_bytes.
 *   - Calls are asynchronous on `stream`.  Arguments are validated on the host
 *     before anything is launched, so a call that returns an error has no
 *     side effect.  Calls on one layer state must be ordered on one stream.
 *   - The kernels are programmatic dependent launches: each may be scheduled
 *     while the previous kernel on the stream drains, and waits for it before
 *     reading what it wrote.  Right after this library's decode compressor (or
 *     top-k) on the same stream and host thread, the decode indexer score (or
 *     the attention's raw-row split) reads data that kernel does not write
 *     before that wait; a kernel of the caller in between is an ordinary
 *     launch, which the next one waits for in full.
 *   - A position `pos` counts tokens already processed by a sequence; token
 *     `pos` is the next one.  Compressed row c of a ratio-r layer pools the
 *     window of tokens c*r .. c*r+r-1 and exists once pos >= (c+1)*r.
 *   - Row-major layouts; "[a][b]" lists the slowest dimension first.
 *   - Kernel-side problems (an exhausted bounded wait) raise a sticky device
 *     error word that ds4c_sync_status reports and clears.
 */
#ifndef DS4C_H
#define DS4C_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define DS4C_API __attribute__((visibility("default")))
#else
#define DS4C_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DS4C_OK = 0,
    DS4C_ERR_NULL = 1,         /* a required pointer is NULL */
    DS4C_ERR_SHAPE = 2,        /* a configuration value outside the supported set */
    DS4C_ERR_CAPACITY = 3,     /* positions past comp_cap*ratio, or an output buffer too small */
    DS4C_ERR_UNSUPPORTED = 4,  /* n_seq > 1 together with n_tok > 1, or a batch above the limit */
    DS4C_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
    DS4C_ERR_DEVICE = 6,       /* a kernel reported a failure through the device error word */
    DS4C_ERR_WORKSPACE = 7     /* workspace NULL or smaller than ds4c_workspace_bytes */
} ds4c_status;

enum { DS4C_F32 = 0, DS4C_BF16 = 1 };

/* One layer's shape.  [P2] §1 (ratio 0, 4 or 128 per layer), §2 (swa: raw
 * ring rows, 128 on Flash), §6 (indexer head_dim 128, top-k 512), §8
 * (head_dim 512 with the last n_rot = 64 dims rotated; compressed layers use
 * their own RoPE base).
 * Supported: ratio in {0,4,128}; head_dim and idx_head_dim in {64,128,256,512};
 * n_rot a multiple of 4, 4 <= n_rot <= min(head_dim, idx_head_dim), at most 128;
 * d_model a multiple of 8; n_heads a multiple of 8, at most 128;
 * 1 <= swa <= 1024; 1 <= top_k <= 2048; idx_cap <= 40960. */
typedef struct {
    uint32_t d_model;       /* hidden width fed to the projections */
    uint32_t head_dim;      /* D: width of a raw / compressed attention row (K = V = the row) */
    uint32_t n_rot;         /* R: RoPE tail width */
    uint32_t idx_head_dim;  /* d: indexer row width (ratio-4 layers) */
    uint32_t n_heads;       /* H: query heads sharing the single KV row */
    uint32_t ratio;         /* 0, 4 or 128 */
    uint32_t swa;           /* raw ring rows S */
    uint32_t top_k;         /* k: compressed rows an attention query keeps (ratio 4) */
    uint32_t comp_cap;      /* attention compressed rows per sequence */
    uint32_t idx_cap;       /* indexer compressed rows per sequence (ratio 4) */
    uint32_t dtype;         /* DS4C_F32 or DS4C_BF16: element type of weights and hidden */
    float rms_eps;          /* RMSNorm epsilon */
    float attn_scale;       /* logit scale, 1/sqrt(head_dim) in the shipped configs */
    float rope_base;        /* compressed-layer RoPE base; theta_i = base^(-2i/n_rot) */
    uint32_t idx_heads;     /* ratio 4: indexer query heads of ds4c_indexer_topk_heads ([P2] §6: 64), 0 if unused */
    uint32_t idx_qat;       /* ratio 4: 1 = the indexer rows (and the heads' queries) take the Hadamard + FP4
                               round trip of [P2] §9; requires idx_head_dim 64 or 128.  0 = identity */
} ds4c_layer_cfg;

/* One compressor lane's weights ([P2] §4, §6: the attention lane and, on
 * ratio-4 layers, the indexer lane with its own ape/kv/gate/norm tensors).
 * With Dl = head_dim (attention lane) or idx_head_dim (indexer lane) and
 * coff = 2 on ratio-4 layers, 1 otherwise:
 *   wkv, wgate: [coff*Dl][d_model] of cfg->dtype;
 *   ape:        [ratio][coff*Dl] float, row pos % ratio is added to the score;
 *   norm:       [Dl] float RMSNorm gain, or NULL for ones. */
typedef struct {
    const void *wkv;
    const void *wgate;
    const float *ape;
    const float *norm;
} ds4c_lane_weights;

/* One lane's state for n_seq sequences ([P2] §2 ds4_layer_cache: compressed
 * rows plus the frontier state_kv / state_score):
 *   comp:        [n_seq][cap][Dl]  appended compressed rows (cap = comp_cap or idx_cap);
 *   state_kv:    [n_seq][coff*ratio][coff*Dl]  frontier (ratio 4: rows 0..3 previous
 *                window, rows 4..7 current window, [P2] §5);
 *   state_score: same shape, scores with the APE already added;
 *   prequant:    optional [n_seq][cap][Dl]: each compressed row as it was before the
 *                FP8 round trip (inspection output), NULL = not written;
 *   comp_split:  attention lane only: [n_seq][cap][2][Dl] bfloat16 (uint16 bits),
 *                hi = bf16(row) and lo = bf16(row - hi) of every appended row, written
 *                by the compress calls next to comp and read by the tensor-core
 *                attention (derived data: not part of the checkpoint).  Required when
 *                ds4c_attn_uses_tensor_cores(cfg) is 1, ignored (may be NULL)
 *                otherwise and on the indexer lane. */
typedef struct {
    float *comp;
    float *state_kv;
    float *state_score;
    float *prequant;
    uint16_t *comp_split;
} ds4c_lane_state;

/* A layer's state: raw: [n_seq][swa][head_dim] ring, slot p % swa holds the raw
 * row of position p ([P2] §2 raw_kv).  idx is unused unless ratio == 4.
 * Calls with n_seq == 1 treat the pointers as the one sequence they address. */
typedef struct {
    float *raw;
    ds4c_lane_state attn;
    ds4c_lane_state idx;
} ds4c_layer_state;

/* 1 when ds4c_sparse_swa_attn runs on the tensor cores for this shape
 * (ratio 0/4/128 with any n_heads: 64 per launch, fewer padded to 64 rows of
 * the MMA tile, more than 64 as groups of 64 that each read the rows again),
 * head_dim in {128, 256, 512}, swa <= 128 (a shorter window masks the older rows
 * of the 128-row raw tile),
 * and top_k <= 512 on ratio-4 layers), 0 when it runs on the CUDA cores.  On
 * the tensor-core path the attention lane's comp_split mirror must be
 * allocated. */
DS4C_API int ds4c_attn_uses_tensor_cores(const ds4c_layer_cfg *cfg);

/* Bytes of workspace that serves every call on `cfg` with prefill chunks of
 * at most max_tok tokens and decode steps of at most max_seq sequences (0: no
 * decode steps).  Returns 0 for an invalid cfg. */
DS4C_API size_t ds4c_workspace_bytes(const ds4c_layer_cfg *cfg, uint32_t max_tok, uint32_t max_seq);

/* Fresh state for n_seq sequences: frontier kv = 0 and score = -inf (so rows
 * no token wrote carry no pooling weight), raw ring zeroed.  Compressed rows
 * are left as they are. */
DS4C_API ds4c_status ds4c_state_init(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                            uint32_t n_seq, cudaStream_t stream);

/* Compressor over n_tok tokens of one sequence at absolute positions
 * pos0 .. pos0+n_tok-1 ([P2] §3 chunked prefill with absolute-position
 * boundaries; §4 compressor_decode_one; §5 ratio-4 frontier and shift; §8
 * tail RoPE; §9 FP8 round trip).  hidden: [n_tok][d_model] of cfg->dtype.
 * idx must be non-NULL exactly when ratio == 4.  Appends rows
 * pos0/ratio .. (pos0+n_tok)/ratio - 1 of each lane and leaves the frontier as
 * the token-by-token recurrence would.  Ratio 0: nothing to do, returns OK.
 * Errors: DS4C_ERR_CAPACITY when (pos0+n_tok)/ratio exceeds a lane's cap. */
DS4C_API ds4c_status ds4c_compress_prefill(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                  const ds4c_lane_weights *idx, const ds4c_layer_state *state,
                                  const void *hidden, uint32_t n_tok, uint64_t pos0,
                                  void *ws, size_t ws_bytes, cudaStream_t stream);

/* Measurement helper, not a step of the path: ds4c_compress_prefill with
 * `after_projection` (a CUDA event, required) recorded on `stream` between the
 * projection GEMM and the fused compressor kernel, so that a caller can time
 * the two apart with events of its own before and after the call.  Same
 * arguments, checks and results as ds4c_compress_prefill otherwise. */
DS4C_API ds4c_status ds4c_compress_prefill_timed(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                                 const ds4c_lane_weights *idx, const ds4c_layer_state *state,
                                                 const void *hidden, uint32_t n_tok, uint64_t pos0, void *ws,
                                                 size_t ws_bytes, cudaEvent_t after_projection, cudaStream_t stream);

/* Compressor for one token of each of n_seq independent sequences, sequence b
 * at position pos_h[b] (host array).  hidden: [n_seq][d_model].  n_seq <= 1024. */
DS4C_API ds4c_status ds4c_compress_decode_step(const ds4c_layer_cfg *cfg, const ds4c_lane_weights *attn,
                                      const ds4c_lane_weights *idx, const ds4c_layer_state *state,
                                      const void *hidden, const uint64_t *pos_h, uint32_t n_seq,
                                      void *ws, size_t ws_bytes, cudaStream_t stream);

/* Indexer top-k of a ratio-4 layer ([P2] §6, §7).  Queries: either n_tok
 * tokens of one sequence at pos_h[0] .. pos_h[0]+n_tok-1 (n_seq == 1), or one
 * token per sequence at pos_h[b] (n_tok == 1).  q_idx: [n][idx_head_dim]
 * float, n = n_seq*n_tok.  A query at position t scores rows c < (t+1)/4 of
 * its sequence's index_comp_kv with s = fmaf chain over i = 0..d-1 of
 * q[i]*row[i] (float, in order) and keeps the top_k largest (ties: lower
 * index), written to topk [n][top_k] in ascending index order, padded with -1.
 * scores (optional, NULL = not written): [n][score_stride] floats, column c
 * valid for c < (t+1)/4; score_stride >= max over queries of (t+1)/4. */
DS4C_API ds4c_status ds4c_indexer_topk(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                              const float *q_idx, const uint64_t *pos_h, uint32_t n_seq,
                              uint32_t n_tok, int32_t *topk, float *scores, size_t score_stride,
                              void *ws, size_t ws_bytes, cudaStream_t stream);

/* Multi-head indexer top-k of a ratio-4 layer with cfg->idx_heads = H_i >= 1
 * heads ([P2] §6: 64 indexer heads of width 128 score the compressed rows; §9:
 * the indexer queries take the same Hadamard + FP4 round trip as the rows when
 * cfg->idx_qat is 1).  Query layout as ds4c_indexer_topk; q_idx: [n][H_i]
 * [idx_head_dim] float, the heads' query vectors before the round trip; w_idx:
 * [n][H_i] float, per-query head weights.  The score of row c for a query is
 * s = 0; for j = 0 .. H_i-1: s = fmaf(w[j], max(dot_j, 0), s), dot_j the in-order
 * fmaf chain of head j's (round-tripped) vector with the row (the pages give no
 * combine; this is the library's reading), then the top_k largest as
 * ds4c_indexer_topk.  Requires idx_head_dim 64 or 128.  Workspace as
 * ds4c_workspace_bytes (it includes the round-tripped query vectors). */
DS4C_API ds4c_status ds4c_indexer_topk_heads(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                                             const float *q_idx, const float *w_idx, const uint64_t *pos_h,
                                             uint32_t n_seq, uint32_t n_tok, int32_t *topk, float *scores,
                                             size_t score_stride, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Sparse sliding-window attention ([P2] §7 indexed mixed attention): for each
 * query at position t and head h, one softmax over the raw rows of positions
 * max(0, t+1-swa) .. t and the compressed rows: ratio 4 the topk list (entries
 * < 0 skipped, the first entry >= (t+1)/4 ends the list), ratio 128 every row
 * c < (t+1)/128, ratio 0 none.  logit = (q . row) * attn_scale; out = sum p*row.
 * Query layout as ds4c_indexer_topk; q: [n][n_heads][head_dim] float (already
 * rotated); raw_new: [n][head_dim] float, the raw rows of the queries' own
 * positions; positions before pos_h[.] come from the ring.  out: [n][n_heads]
 * [head_dim] float.  commit_ring != 0 then writes raw_new into the ring (the
 * last min(n_tok, swa) rows of a chunk; one row per sequence in a decode
 * step), after the attention has read it.  topk may be NULL unless ratio == 4. */
DS4C_API ds4c_status ds4c_sparse_swa_attn(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                                 const float *q, const float *raw_new, const int32_t *topk,
                                 const uint64_t *pos_h, uint32_t n_seq, uint32_t n_tok,
                                 float *out, int commit_ring, void *ws, size_t ws_bytes,
                                 cudaStream_t stream);

/* Score capacity of ds4c_indexer_topk_noalloc: 2M floats (8 MiB). */
#define DS4C_NOALLOC_SCORE_FLOATS (2u * 1024u * 1024u)

/* ds4c_indexer_topk for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment variant of the indexer call.
 * Some callers cannot call cudaMalloc or hand over a workspace: runtimes that
 * own all device memory through their own pool and forbid allocation on the
 * serving path (an allocation can synchronise the device or fragment the
 * pool), or code running where no allocator is reachable.  This call takes
 * the same arguments and gives the same result as ds4c_indexer_topk with
 * scores = NULL, but keeps its score matrix in a fixed file-scope device array
 * of DS4C_NOALLOC_SCORE_FLOATS floats instead of the caller's workspace.
 *   - Limit: n_seq * n_tok * round_up((last query position + 1) / 4, 4) must not
 *     exceed DS4C_NOALLOC_SCORE_FLOATS, otherwise DS4C_ERR_CAPACITY and nothing
 *     is launched (e.g. a 32-sequence decode step at 65536 context fits; a
 *     4096-token prefill chunk at 131072 context does not).
 *   - The array exists on every GPU that loads the library, until the process
 *     exits.  The first call on a device looks up the array's device address
 *     (with that device current) and keeps it; make that first call before any
 *     stream capture.  The kept address does not survive cudaDeviceReset: do
 *     not call this entry point on a device after resetting it.
 *   - Every call shares the array: calls whose kernels overlap on the GPU (on
 *     streams without ordering between them) race on it.  A call reads only
 *     scores it wrote itself, so no part of the array needs clearing.
 *   - It allocates nothing and calls no allocating library routine. */
DS4C_API ds4c_status ds4c_indexer_topk_noalloc(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                                               const float *q_idx, const uint64_t *pos_h, uint32_t n_seq,
                                               uint32_t n_tok, int32_t *topk, cudaStream_t stream);

/* Floats of one sequence's checkpoint after pos tokens:
 *   min(pos, swa)*D + [ratio != 0] ((pos/ratio)*D + 2*(coff*ratio)*(coff*D))
 *   + [ratio == 4] ((pos/4)*d + 2*8*(2d)). */
DS4C_API size_t ds4c_checkpoint_floats(const ds4c_layer_cfg *cfg, uint64_t pos);

/* Logical-order checkpoint of sequence `seq` after pos tokens into dst ([P1]
 * §5 payload body order, §6 the raw ring written in logical position order,
 * §7 frontier tensors): raw rows of positions pos-n_live .. pos-1 (n_live =
 * min(pos, swa)), attn comp rows 0 .. pos/ratio-1, attn state_kv, attn
 * state_score, then on ratio-4 layers idx comp rows 0 .. pos/4-1, idx
 * state_kv, idx state_score.  Bit copy.  dst_floats < ds4c_checkpoint_floats
 * -> DS4C_ERR_CAPACITY.  *written_h (host, optional) receives the count. */
DS4C_API ds4c_status ds4c_checkpoint_gather(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                                   uint32_t seq, uint64_t pos, float *dst, size_t dst_floats,
                                   size_t *written_h, cudaStream_t stream);

/* Restore of a checkpoint into sequence `seq` of `state`: the inverse of
 * ds4c_checkpoint_gather on a buffer in the same layout ([P1] §6: the raw rows,
 * saved in logical position order, go back in order into the live ring, slot
 * p % swa for position p; §7: the compressed rows and both lanes' frontier
 * tensors, so that compression continues exactly from pos).  Rows of comp past
 * the live count and ring slots past min(pos, swa) live rows are left as they
 * are.  On the tensor-core attention path the attention lane's comp_split
 * mirror of the restored rows is rebuilt as well.  src (device) holds
 * ds4c_checkpoint_floats(cfg, pos) floats; fewer -> DS4C_ERR_CAPACITY. */
DS4C_API ds4c_status ds4c_checkpoint_scatter(const ds4c_layer_cfg *cfg, const ds4c_layer_state *state,
                                             uint32_t seq, uint64_t pos, const float *src, size_t src_floats,
                                             cudaStream_t stream);

/* The fixed header of the DSV4 session payload ([P1] §5): 13 u32 fields, in
 * order: magic "DSV4" (0x34565344), payload version 2, saved context size,
 * prefill chunk size, raw KV ring capacity, raw sliding-window length,
 * compressed KV capacity, checkpoint token count, layer count, raw/head KV
 * dimension, indexer head dimension, vocabulary size, live raw rows serialised
 * in the body.  The body that follows it is, in order: the token ids, the
 * next-token logits, per-layer compressed-row counts (attention, then ratio-4
 * indexer; pos / ratio each), then the per-layer data ds4c_checkpoint_gather
 * writes.  Host only. */
#define DS4C_PAYLOAD_MAGIC 0x34565344u
#define DS4C_PAYLOAD_VERSION 2u
#define DS4C_PAYLOAD_U32_FIELDS 13u
typedef struct {
    uint32_t ctx_size, prefill_chunk, raw_cap, raw_window, comp_cap, token_count, layer_count, head_dim,
        idx_head_dim, vocab_size, live_raw_rows;
} ds4c_payload_info;
DS4C_API ds4c_status ds4c_payload_header(const ds4c_payload_info *info, uint32_t out[DS4C_PAYLOAD_U32_FIELDS]);

/* Bytes of the DSV4 payload ([P1] §5) of a stack of n_layers layers (cfgs[l],
 * layer order) after pos tokens with a vocabulary of vocab_size logits:
 * 4 * (13 + pos + vocab_size + 2 * n_layers) + 4 * sum over layers of
 * ds4c_checkpoint_floats(cfgs[l], pos).  0 for an invalid cfg or n_layers == 0. */
DS4C_API size_t ds4c_payload_bytes(const ds4c_layer_cfg *cfgs, uint32_t n_layers, uint64_t pos, uint32_t vocab_size);

/* Writes sequence `seq` of a layer stack as one DSV4 payload into the device
 * buffer dst ([P1] §5 body order; §6 raw rows in logical position order; §7 the
 * frontier tensors): the header of `info` (info->token_count is the checkpoint
 * position pos, info->layer_count == n_layers, info->live_raw_rows ==
 * min(pos, raw_window)), the pos token ids tokens_h (host), the vocab_size logits
 * logits_h (host; both come from outside this path), the attention row counts
 * pos / ratio (0 on ratio-0 layers) and the indexer row counts pos / 4 (ratio-4
 * layers, else 0) as u32 per layer, then for each layer in order the body
 * ds4c_checkpoint_gather writes.  cfgs[l] / states[l] describe layer l: every
 * layer's swa must equal raw_window and raw_cap, its head_dim the header's, a
 * ratio-4 layer's idx_head_dim the header's, and its comp_cap must not exceed
 * the header's comp_cap (else DS4C_ERR_SHAPE).  dst must be 16-byte aligned
 * and hold ds4c_payload_bytes bytes (else DS4C_ERR_CAPACITY); *written_h (host,
 * optional) receives that count.  The host fields are staged before the call
 * returns; the copies and kernels run on `stream`. */
DS4C_API ds4c_status ds4c_payload_write(const ds4c_payload_info *info, const ds4c_layer_cfg *cfgs,
                                        const ds4c_layer_state *states, uint32_t n_layers, uint32_t seq,
                                        const uint32_t *tokens_h, const float *logits_h, void *dst, size_t dst_bytes,
                                        size_t *written_h, cudaStream_t stream);

/* Restores sequence `seq` of a layer stack from a DSV4 payload in the device
 * buffer src, the inverse of ds4c_payload_write.  The payload's header must
 * match `expect` in every field but the token count and the live raw rows
 * (a payload written for another runtime shape is refused with
 * DS4C_ERR_SHAPE, as is a live-row count or a per-layer row count that
 * disagrees with the token count); then each layer's body is scattered into
 * states[l] (ds4c_checkpoint_scatter), the token ids are copied to tokens_h
 * (host, room for tokens_cap ids, else DS4C_ERR_CAPACITY), the logits to
 * logits_h (host, expect->vocab_size floats) and the token count to
 * *token_count_h.  The header and the host fields are read synchronously
 * (the call synchronises `stream` twice); nothing is written before every
 * check has passed. */
DS4C_API ds4c_status ds4c_payload_read(const ds4c_payload_info *expect, const ds4c_layer_cfg *cfgs,
                                       const ds4c_layer_state *states, uint32_t n_layers, uint32_t seq,
                                       const void *src, size_t src_bytes, uint32_t *tokens_h, size_t tokens_cap,
                                       float *logits_h, uint32_t *token_count_h, cudaStream_t stream);

/* Measurement helper, not a step of the path: the fp32 FMA rate of the GPU,
 * the denominator of the indexer score's roofline (an in-order fp32 fmaf chain
 * per output on the CUDA cores).  Launches `blocks` CTAs of 256 threads, each
 * thread running independent fmaf chains for `iters` rounds in registers and
 * storing one float to out[blocks * 256] (device, caller-owned, 4-byte
 * aligned); *flops_h (host) receives the launch's flop count.  The caller
 * times the launch on `stream`.  DS4C_ERR_NULL / DS4C_ERR_SHAPE (blocks or
 * iters zero, iters above 2^24, misaligned out) before any launch. */
DS4C_API ds4c_status ds4c_fma_probe(uint32_t blocks, uint32_t iters, float *out, double *flops_h,
                                    cudaStream_t stream);

/* Test hooks of the failure path (not steps of the method).  Every spin-wait in
 * the kernels (an mbarrier wait for copies or MMAs) is bounded: when its limit
 * runs out the kernel raises a sticky device error word, waits (bounded again)
 * for what it still has in flight, frees its tensor memory and returns, so the
 * context stays usable and ds4c_sync_status reports DS4C_ERR_DEVICE.
 * ds4c_test_set_wait_limit sets that limit on the current device (0 = the
 * default of 4 s); ds4c_test_wait_timeout launches one CTA that waits, bounded
 * by limit_ns, on an mbarrier nothing arrives on, through the same wait routine
 * as the indexer kernels, so its limit runs out and it raises the indexer's
 * error word (no fault, no hang). */
DS4C_API ds4c_status ds4c_test_set_wait_limit(uint64_t limit_ns);
DS4C_API ds4c_status ds4c_test_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/* Synchronises `stream`, then reports (and clears) the device error word:
 * DS4C_ERR_DEVICE if a kernel raised it, DS4C_ERR_CUDA if the stream failed. */
DS4C_API ds4c_status ds4c_sync_status(cudaStream_t stream);

/* Static description of a status code. */
DS4C_API const char *ds4c_status_string(ds4c_status status);

/* Name of the CUDA runtime error behind the calling thread's most recent
 * DS4C_ERR_CUDA ("cudaSuccess" if there was none), for diagnostics. */
DS4C_API const char *ds4c_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DS4C_H */
