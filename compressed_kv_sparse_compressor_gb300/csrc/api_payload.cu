// DSV4 session payload of a layer stack, "【#4】ds4.c を読み解く" §5-§7: the
// 13-field header, the checkpoint token ids, the next-token logits, two u32
// row counts per layer (attention compressed rows, ratio-4 indexer rows), then
// each layer's body in layer order: its raw SWA rows in logical position
// order, its attention compressed rows and compressor frontier, and on ratio-4
// layers its indexer rows and indexer frontier (the body ds4c_checkpoint_gather
// writes for one layer).  The payload lives in a device buffer; the host-side
// fields are copied in and out with cudaMemcpyAsync, the layer bodies are
// moved by the gather / scatter kernels.
#include <string.h>

#include <vector>

#include "ds4c_internal.cuh"

using namespace ds4c;

namespace {

constexpr size_t kHeaderBytes = 4 * DS4C_PAYLOAD_U32_FIELDS;

uint32_t attn_rows(const ds4c_layer_cfg &c, uint64_t pos) { return c.ratio ? (uint32_t)(pos / c.ratio) : 0u; }
uint32_t idx_rows(const ds4c_layer_cfg &c, uint64_t pos) { return c.ratio == 4 ? (uint32_t)(pos / 4) : 0u; }

// Byte offset of layer 0's body.
size_t body_offset(uint64_t token_count, uint32_t vocab, uint32_t n_layers) {
    return kHeaderBytes + 4 * ((size_t)token_count + vocab + 2 * (size_t)n_layers);
}

// Header fields the stack's configurations fix: every layer has the ring,
// window and head widths the header states; ratio-4 layers the indexer width;
// no layer holds more compressed rows than the header's capacity.
ds4c_status check_stack(const ds4c_payload_info &h, const ds4c_layer_cfg *cfgs, uint32_t n_layers) {
    if (h.layer_count != n_layers || n_layers == 0) return DS4C_ERR_SHAPE;
    for (uint32_t l = 0; l < n_layers; l++) {
        const ds4c_layer_cfg &c = cfgs[l];
        const ds4c_status s = check_cfg(&c);
        if (s != DS4C_OK) return s;
        if (c.swa != h.raw_window || c.swa != h.raw_cap || c.head_dim != h.head_dim) return DS4C_ERR_SHAPE;
        if (c.ratio == 4 && c.idx_head_dim != h.idx_head_dim) return DS4C_ERR_SHAPE;
        if (c.ratio != 0 && c.comp_cap > h.comp_cap) return DS4C_ERR_SHAPE;
    }
    return DS4C_OK;
}

size_t stack_bytes(const ds4c_layer_cfg *cfgs, uint32_t n_layers, uint64_t pos, uint32_t vocab) {
    size_t total = body_offset(pos, vocab, n_layers);
    for (uint32_t l = 0; l < n_layers; l++) total += 4 * ds4c_checkpoint_floats(&cfgs[l], pos);
    return total;
}

}  // namespace

extern "C" {

size_t ds4c_payload_bytes(const ds4c_layer_cfg *cfgs, uint32_t n_layers, uint64_t pos, uint32_t vocab_size) {
    if (!cfgs || n_layers == 0) return 0;
    for (uint32_t l = 0; l < n_layers; l++)
        if (check_cfg(&cfgs[l]) != DS4C_OK) return 0;
    return stack_bytes(cfgs, n_layers, pos, vocab_size);
}

ds4c_status ds4c_payload_write(const ds4c_payload_info *info, const ds4c_layer_cfg *cfgs,
                               const ds4c_layer_state *states, uint32_t n_layers, uint32_t seq,
                               const uint32_t *tokens_h, const float *logits_h, void *dst, size_t dst_bytes,
                               size_t *written_h, cudaStream_t stream) {
    if (!info || !cfgs || !states || !dst) return DS4C_ERR_NULL;
    const ds4c_payload_info &h = *info;
    if ((h.token_count && !tokens_h) || (h.vocab_size && !logits_h)) return DS4C_ERR_NULL;
    ds4c_status s = check_stack(h, cfgs, n_layers);
    if (s != DS4C_OK) return s;
    const uint64_t pos = h.token_count;
    if (h.live_raw_rows != (pos < h.raw_window ? pos : h.raw_window)) return DS4C_ERR_SHAPE;
    if (((uintptr_t)dst & 15) != 0) return DS4C_ERR_SHAPE;
    for (uint32_t l = 0; l < n_layers; l++) {
        const ds4c_layer_cfg &c = cfgs[l];
        if (c.ratio != 0 && attn_rows(c, pos) > c.comp_cap) return DS4C_ERR_CAPACITY;
        if (c.ratio == 4 && idx_rows(c, pos) > c.idx_cap) return DS4C_ERR_CAPACITY;
    }
    const size_t need = stack_bytes(cfgs, n_layers, pos, h.vocab_size);
    if (dst_bytes < need) return DS4C_ERR_CAPACITY;
    // host part: header, token ids, logits, the two count arrays (one staging buffer, one copy)
    const size_t off0 = body_offset(pos, h.vocab_size, n_layers);
    std::vector<uint32_t> head(off0 / 4);
    ds4c_payload_header(info, head.data());
    size_t w = DS4C_PAYLOAD_U32_FIELDS;
    if (pos) memcpy(&head[w], tokens_h, 4 * (size_t)pos);
    w += (size_t)pos;
    if (h.vocab_size) memcpy(&head[w], logits_h, 4 * (size_t)h.vocab_size);
    w += h.vocab_size;
    for (uint32_t l = 0; l < n_layers; l++) head[w + l] = attn_rows(cfgs[l], pos);
    for (uint32_t l = 0; l < n_layers; l++) head[w + n_layers + l] = idx_rows(cfgs[l], pos);
    // pageable source: the copy has been staged when the call returns, so the vector may go
    cudaError_t e = cudaMemcpyAsync(dst, head.data(), off0, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_status(e);
    size_t off = off0;
    for (uint32_t l = 0; l < n_layers; l++) {
        const size_t nf = ds4c_checkpoint_floats(&cfgs[l], pos);
        float *body = reinterpret_cast<float *>(static_cast<char *>(dst) + off);
        s = ds4c_checkpoint_gather(&cfgs[l], &states[l], seq, pos, body, nf, nullptr, stream);
        if (s != DS4C_OK) return s;
        off += 4 * nf;
    }
    if (written_h) *written_h = off;
    return DS4C_OK;
}

ds4c_status ds4c_payload_read(const ds4c_payload_info *expect, const ds4c_layer_cfg *cfgs,
                              const ds4c_layer_state *states, uint32_t n_layers, uint32_t seq, const void *src,
                              size_t src_bytes, uint32_t *tokens_h, size_t tokens_cap, float *logits_h,
                              uint32_t *token_count_h, cudaStream_t stream) {
    if (!expect || !cfgs || !states || !src || !token_count_h) return DS4C_ERR_NULL;
    if (expect->vocab_size && !logits_h) return DS4C_ERR_NULL;
    if (((uintptr_t)src & 15) != 0) return DS4C_ERR_SHAPE;
    ds4c_status s = check_stack(*expect, cfgs, n_layers);
    if (s != DS4C_OK) return s;
    if (src_bytes < kHeaderBytes) return DS4C_ERR_CAPACITY;
    uint32_t hdr[DS4C_PAYLOAD_U32_FIELDS];
    cudaError_t e = cudaMemcpyAsync(hdr, src, kHeaderBytes, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_status(e);
    // a payload written for another runtime shape is refused ([P3]: the header rejects a
    // file of a different payload ABI): every field but the token and live-row counts
    uint32_t want[DS4C_PAYLOAD_U32_FIELDS];
    ds4c_payload_header(expect, want);
    for (unsigned i = 0; i < DS4C_PAYLOAD_U32_FIELDS; i++) {
        if (i == 7 || i == 12) continue;                 // token_count, live_raw_rows
        if (hdr[i] != want[i]) return DS4C_ERR_SHAPE;
    }
    const uint64_t pos = hdr[7];
    if (hdr[12] != (pos < expect->raw_window ? pos : expect->raw_window)) return DS4C_ERR_SHAPE;
    if (pos > tokens_cap || (pos && !tokens_h)) return DS4C_ERR_CAPACITY;
    for (uint32_t l = 0; l < n_layers; l++) {
        const ds4c_layer_cfg &c = cfgs[l];
        if (c.ratio != 0 && attn_rows(c, pos) > c.comp_cap) return DS4C_ERR_CAPACITY;
        if (c.ratio == 4 && idx_rows(c, pos) > c.idx_cap) return DS4C_ERR_CAPACITY;
    }
    const size_t need = stack_bytes(cfgs, n_layers, pos, expect->vocab_size);
    if (src_bytes < need) return DS4C_ERR_CAPACITY;
    const size_t off0 = body_offset(pos, expect->vocab_size, n_layers);
    std::vector<uint32_t> head(off0 / 4);
    e = cudaMemcpyAsync(head.data(), src, off0, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_status(e);
    // the per-layer row counts must be the ones the token count implies
    size_t w = DS4C_PAYLOAD_U32_FIELDS + (size_t)pos + expect->vocab_size;
    for (uint32_t l = 0; l < n_layers; l++)
        if (head[w + l] != attn_rows(cfgs[l], pos) || head[w + n_layers + l] != idx_rows(cfgs[l], pos))
            return DS4C_ERR_SHAPE;
    size_t off = off0;
    for (uint32_t l = 0; l < n_layers; l++) {
        const size_t nf = ds4c_checkpoint_floats(&cfgs[l], pos);
        const float *body = reinterpret_cast<const float *>(static_cast<const char *>(src) + off);
        s = ds4c_checkpoint_scatter(&cfgs[l], &states[l], seq, pos, body, nf, stream);
        if (s != DS4C_OK) return s;
        off += 4 * nf;
    }
    if (pos) memcpy(tokens_h, &head[DS4C_PAYLOAD_U32_FIELDS], 4 * (size_t)pos);
    if (expect->vocab_size) memcpy(logits_h, &head[DS4C_PAYLOAD_U32_FIELDS + pos], 4 * (size_t)expect->vocab_size);
    *token_count_h = (uint32_t)pos;
    return DS4C_OK;
}

}  // extern "C"
