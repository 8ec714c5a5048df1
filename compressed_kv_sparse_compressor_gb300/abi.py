"""ctypes binding of libds4c (include/ds4c.h): the same names, argument
marshalling only.  Every step of the path runs in the library's kernels; this
module never computes any part of it and has no fallback: if the shared
library is missing or fails to load, every call raises."""

from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libds4c.so")

DS4C_OK = 0
DS4C_ERR_NULL = 1
DS4C_ERR_SHAPE = 2
DS4C_ERR_CAPACITY = 3
DS4C_ERR_UNSUPPORTED = 4
DS4C_ERR_CUDA = 5
DS4C_ERR_DEVICE = 6
DS4C_ERR_WORKSPACE = 7
DS4C_F32 = 0
DS4C_BF16 = 1

EXPORTS = (
    "ds4c_workspace_bytes", "ds4c_state_init", "ds4c_compress_prefill", "ds4c_compress_decode_step",
    "ds4c_indexer_topk", "ds4c_sparse_swa_attn", "ds4c_checkpoint_floats", "ds4c_checkpoint_gather",
    "ds4c_sync_status", "ds4c_status_string", "ds4c_last_cuda_error", "ds4c_attn_uses_tensor_cores",
    "ds4c_indexer_topk_noalloc", "ds4c_checkpoint_scatter", "ds4c_payload_header", "ds4c_fma_probe",
    "ds4c_payload_bytes", "ds4c_payload_write", "ds4c_payload_read", "ds4c_compress_prefill_timed",
    "ds4c_indexer_topk_heads", "ds4c_test_set_wait_limit", "ds4c_test_wait_timeout",
)
PAYLOAD_U32_FIELDS = 13
NOALLOC_SCORE_FLOATS = 2 * 1024 * 1024


class Ds4cError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: status {status} ({status_string(status)})"
        if status == DS4C_ERR_CUDA:
            msg += f" [{lib().ds4c_last_cuda_error().decode()}]"
        super().__init__(msg)


class LayerCfg(C.Structure):
    _fields_ = [("d_model", C.c_uint32), ("head_dim", C.c_uint32), ("n_rot", C.c_uint32),
                ("idx_head_dim", C.c_uint32), ("n_heads", C.c_uint32), ("ratio", C.c_uint32),
                ("swa", C.c_uint32), ("top_k", C.c_uint32), ("comp_cap", C.c_uint32),
                ("idx_cap", C.c_uint32), ("dtype", C.c_uint32), ("rms_eps", C.c_float),
                ("attn_scale", C.c_float), ("rope_base", C.c_float), ("idx_heads", C.c_uint32),
                ("idx_qat", C.c_uint32)]


class LaneWeights(C.Structure):
    _fields_ = [("wkv", C.c_void_p), ("wgate", C.c_void_p), ("ape", C.c_void_p), ("norm", C.c_void_p)]


class PayloadInfo(C.Structure):
    _fields_ = [(n, C.c_uint32) for n in ("ctx_size", "prefill_chunk", "raw_cap", "raw_window", "comp_cap",
                                           "token_count", "layer_count", "head_dim", "idx_head_dim", "vocab_size",
                                           "live_raw_rows")]


class LaneState(C.Structure):
    _fields_ = [("comp", C.c_void_p), ("state_kv", C.c_void_p), ("state_score", C.c_void_p),
                ("prequant", C.c_void_p), ("comp_split", C.c_void_p)]


class LayerState(C.Structure):
    _fields_ = [("raw", C.c_void_p), ("attn", LaneState), ("idx", LaneState)]


_lib = None


def lib() -> C.CDLL:
    """Load libds4c.so (built by build.py); raise if it is not there."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libds4c.so not built ({LIB_PATH}); run compressed_kv_sparse_compressor_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    P, U32, U64, SZ = C.c_void_p, C.c_uint32, C.c_uint64, C.c_size_t
    cfgp, lwp, lsp = C.POINTER(LayerCfg), C.POINTER(LaneWeights), C.POINTER(LayerState)
    st = C.c_int
    sig = {
        "ds4c_workspace_bytes": (SZ, [cfgp, U32, U32]),
        "ds4c_attn_uses_tensor_cores": (C.c_int, [cfgp]),
        "ds4c_state_init": (st, [cfgp, lsp, U32, P]),
        "ds4c_compress_prefill": (st, [cfgp, lwp, lwp, lsp, P, U32, U64, P, SZ, P]),
        "ds4c_compress_prefill_timed": (st, [cfgp, lwp, lwp, lsp, P, U32, U64, P, SZ, P, P]),
        "ds4c_compress_decode_step": (st, [cfgp, lwp, lwp, lsp, P, C.POINTER(U64), U32, P, SZ, P]),
        "ds4c_indexer_topk": (st, [cfgp, lsp, P, C.POINTER(U64), U32, U32, P, P, SZ, P, SZ, P]),
        "ds4c_indexer_topk_heads": (st, [cfgp, lsp, P, P, C.POINTER(U64), U32, U32, P, P, SZ, P, SZ, P]),
        "ds4c_sparse_swa_attn": (st, [cfgp, lsp, P, P, P, C.POINTER(U64), U32, U32, P, C.c_int, P, SZ, P]),
        "ds4c_indexer_topk_noalloc": (st, [cfgp, lsp, P, C.POINTER(U64), U32, U32, P, P]),
        "ds4c_checkpoint_floats": (SZ, [cfgp, U64]),
        "ds4c_checkpoint_gather": (st, [cfgp, lsp, U32, U64, P, SZ, C.POINTER(SZ), P]),
        "ds4c_checkpoint_scatter": (st, [cfgp, lsp, U32, U64, P, SZ, P]),
        "ds4c_payload_header": (st, [C.POINTER(PayloadInfo), C.POINTER(C.c_uint32 * PAYLOAD_U32_FIELDS)]),
        "ds4c_payload_bytes": (SZ, [cfgp, U32, U64, U32]),
        "ds4c_payload_write": (st, [C.POINTER(PayloadInfo), cfgp, lsp, U32, U32, P, P, P, SZ, C.POINTER(SZ), P]),
        "ds4c_payload_read": (st, [C.POINTER(PayloadInfo), cfgp, lsp, U32, U32, P, SZ, P, SZ, P,
                                   C.POINTER(U32), P]),
        "ds4c_fma_probe": (st, [U32, U32, P, C.POINTER(C.c_double), P]),
        "ds4c_test_set_wait_limit": (st, [U64]),
        "ds4c_test_wait_timeout": (st, [U64, P]),
        "ds4c_sync_status": (st, [P]),
        "ds4c_status_string": (C.c_char_p, [C.c_int]),
        "ds4c_last_cuda_error": (C.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def status_string(s: int) -> str:
    return lib().ds4c_status_string(s).decode()


def check(s: int, where: str):
    if s != DS4C_OK:
        raise Ds4cError(s, where)


def u64_array(values):
    vals = [int(v) for v in values]
    return (C.c_uint64 * max(len(vals), 1))(*vals)


# Thin call wrappers with the ABI's names; pointers are ints (device
# addresses), None for NULL.  Each returns the raw status.

def ds4c_workspace_bytes(cfg, max_tok, max_seq=0):
    return lib().ds4c_workspace_bytes(C.byref(cfg), max_tok, max_seq)


def ds4c_attn_uses_tensor_cores(cfg):
    return lib().ds4c_attn_uses_tensor_cores(C.byref(cfg))


def ds4c_state_init(cfg, state, n_seq, stream):
    return lib().ds4c_state_init(C.byref(cfg), C.byref(state), n_seq, stream)


def ds4c_compress_prefill(cfg, attn_w, idx_w, state, hidden, n_tok, pos0, ws, ws_bytes, stream):
    return lib().ds4c_compress_prefill(C.byref(cfg), C.byref(attn_w) if attn_w is not None else None,
                                       C.byref(idx_w) if idx_w is not None else None, C.byref(state),
                                       hidden, n_tok, pos0, ws, ws_bytes, stream)


def ds4c_compress_prefill_timed(cfg, attn_w, idx_w, state, hidden, n_tok, pos0, ws, ws_bytes, event, stream):
    return lib().ds4c_compress_prefill_timed(C.byref(cfg), C.byref(attn_w) if attn_w is not None else None,
                                             C.byref(idx_w) if idx_w is not None else None, C.byref(state),
                                             hidden, n_tok, pos0, ws, ws_bytes, event, stream)


def ds4c_compress_decode_step(cfg, attn_w, idx_w, state, hidden, pos_h, n_seq, ws, ws_bytes, stream):
    return lib().ds4c_compress_decode_step(C.byref(cfg), C.byref(attn_w) if attn_w is not None else None,
                                           C.byref(idx_w) if idx_w is not None else None, C.byref(state),
                                           hidden, pos_h, n_seq, ws, ws_bytes, stream)


def ds4c_indexer_topk(cfg, state, q_idx, pos_h, n_seq, n_tok, topk, scores, score_stride, ws, ws_bytes, stream):
    return lib().ds4c_indexer_topk(C.byref(cfg), C.byref(state), q_idx, pos_h, n_seq, n_tok, topk, scores,
                                   score_stride, ws, ws_bytes, stream)


def ds4c_indexer_topk_heads(cfg, state, q_idx, w_idx, pos_h, n_seq, n_tok, topk, scores, score_stride, ws, ws_bytes,
                            stream):
    return lib().ds4c_indexer_topk_heads(C.byref(cfg), C.byref(state), q_idx, w_idx, pos_h, n_seq, n_tok, topk,
                                         scores, score_stride, ws, ws_bytes, stream)


def ds4c_indexer_topk_noalloc(cfg, state, q_idx, pos_h, n_seq, n_tok, topk, stream):
    return lib().ds4c_indexer_topk_noalloc(C.byref(cfg), C.byref(state), q_idx, pos_h, n_seq, n_tok, topk, stream)


def ds4c_sparse_swa_attn(cfg, state, q, raw_new, topk, pos_h, n_seq, n_tok, out, commit_ring, ws, ws_bytes, stream):
    return lib().ds4c_sparse_swa_attn(C.byref(cfg), C.byref(state), q, raw_new, topk, pos_h, n_seq, n_tok, out,
                                      int(commit_ring), ws, ws_bytes, stream)


def ds4c_checkpoint_floats(cfg, pos):
    return lib().ds4c_checkpoint_floats(C.byref(cfg), pos)


def ds4c_checkpoint_gather(cfg, state, seq, pos, dst, dst_floats, written, stream):
    return lib().ds4c_checkpoint_gather(C.byref(cfg), C.byref(state), seq, pos, dst, dst_floats, written, stream)


def ds4c_checkpoint_scatter(cfg, state, seq, pos, src, src_floats, stream):
    return lib().ds4c_checkpoint_scatter(C.byref(cfg), C.byref(state), seq, pos, src, src_floats, stream)


def ds4c_payload_header(info):
    """The 13 u32 fields of the DSV4 payload header for `info` (a PayloadInfo)."""
    out = (C.c_uint32 * PAYLOAD_U32_FIELDS)()
    check(lib().ds4c_payload_header(C.byref(info), C.byref(out)), "ds4c_payload_header")
    return list(out)


def _stack(cfgs, states=None):
    ca = (LayerCfg * len(cfgs))(*cfgs)
    sa = None if states is None else (LayerState * len(states))(*states)
    return ca, sa


def ds4c_payload_bytes(cfgs, pos, vocab_size):
    ca, _ = _stack(cfgs)
    return lib().ds4c_payload_bytes(ca, len(cfgs), pos, vocab_size)


def ds4c_payload_write(info, cfgs, states, seq, tokens_h, logits_h, dst, dst_bytes, stream):
    """tokens_h / logits_h: host numpy arrays (uint32 / float32).  Returns (status, bytes written)."""
    ca, sa = _stack(cfgs, states)
    w = C.c_size_t(0)
    tp = tokens_h.ctypes.data_as(C.c_void_p) if tokens_h is not None and tokens_h.size else None
    lp = logits_h.ctypes.data_as(C.c_void_p) if logits_h is not None and logits_h.size else None
    s = lib().ds4c_payload_write(C.byref(info), ca, sa, len(cfgs), seq, tp, lp, dst, dst_bytes, C.byref(w), stream)
    return s, w.value


def ds4c_payload_read(expect, cfgs, states, seq, src, src_bytes, tokens_h, logits_h, stream):
    """tokens_h / logits_h: writable host numpy arrays.  Returns (status, token count)."""
    ca, sa = _stack(cfgs, states)
    n = C.c_uint32(0)
    tp = tokens_h.ctypes.data_as(C.c_void_p) if tokens_h is not None and tokens_h.size else None
    lp = logits_h.ctypes.data_as(C.c_void_p) if logits_h is not None and logits_h.size else None
    cap = 0 if tokens_h is None else tokens_h.size
    s = lib().ds4c_payload_read(C.byref(expect), ca, sa, len(cfgs), seq, src, src_bytes, tp, cap, lp, C.byref(n),
                                stream)
    return s, n.value


def ds4c_fma_probe(blocks, iters, out_ptr, stream):
    """Launch the fp32 FMA-rate probe; returns (status, flops of the launch)."""
    fl = C.c_double(0.0)
    s = lib().ds4c_fma_probe(blocks, iters, out_ptr, C.byref(fl), stream)
    return s, fl.value


def ds4c_test_set_wait_limit(limit_ns):
    return lib().ds4c_test_set_wait_limit(limit_ns)


def ds4c_test_wait_timeout(limit_ns, stream):
    return lib().ds4c_test_wait_timeout(limit_ns, stream)


def ds4c_sync_status(stream):
    return lib().ds4c_sync_status(stream)
