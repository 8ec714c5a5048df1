"""ctypes wrapper of the plain-C oracle of the compressed-KV attention path.

TEST INFRASTRUCTURE: only the tests, the package smoke check and the
benchmark's CPU-baseline leg use this module.  It never imports the CUDA
package and takes plain numpy arrays.  ``build()`` compiles ``ds4c_oracle.c``
with gcc (OpenMP, no fast-math, no FMA contraction).
"""

from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ds4c_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libds4c_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (host C only)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Cfg(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("head_dim", C.c_int32), ("n_rot", C.c_int32),
                ("idx_head_dim", C.c_int32), ("n_heads", C.c_int32), ("ratio", C.c_int32),
                ("swa", C.c_int32), ("top_k", C.c_int32), ("comp_cap", C.c_int32),
                ("idx_cap", C.c_int32), ("bf16", C.c_int32), ("rms_eps", C.c_float),
                ("attn_scale", C.c_float), ("rope_base", C.c_double), ("idx_heads", C.c_int32),
                ("idx_qat", C.c_int32)]


class LaneW(C.Structure):
    _fields_ = [("wkv", C.c_void_p), ("wgate", C.c_void_p), ("ape", C.c_void_p), ("norm", C.c_void_p)]


class LaneS(C.Structure):
    _fields_ = [("comp", C.c_void_p), ("state_kv", C.c_void_p), ("state_score", C.c_void_p),
                ("prequant", C.c_void_p)]


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB_PATH)
        P, I, U64, F, D = C.c_void_p, C.c_int, C.c_uint64, C.c_float, C.c_double
        sig = {
            "orc_num_threads": (I, []),
            "orc_layer_ratio": (I, [I, I]),
            "orc_raw_cap": (I, [I]),
            "orc_prefill_chunk": (I, [I, I]),
            "orc_inv_freq": (None, [D, I, P]),
            "orc_project": (None, [P, P, I, I, I, I, P]),
            "orc_e4m3_rne": (F, [F]),
            "orc_fp8_scale_exp": (I, [F]),
            "orc_fp8_roundtrip": (None, [P, I]),
            "orc_rope_tail": (None, [P, I, I, U64, P]),
            "orc_rmsnorm": (None, [P, I, P, F]),
            "orc_compress_token": (None, [P, I, P, P, P, LaneS, P, P, U64]),
            "orc_state_init_lane": (None, [P, I, LaneS]),
            "orc_compress": (None, [P, P, P, LaneS, LaneS, P, I, U64, P]),
            "orc_index_score": (F, [P, P, I]),
            "orc_topk": (None, [P, I, I, P]),
            "orc_indexer_topk": (None, [P, P, P, P, I, P, P, C.c_int64]),
            "orc_attention": (None, [P, P, P, P, P, P, U64, I, P]),
            "orc_ring_commit": (None, [P, P, P, U64, I]),
            "orc_checkpoint_floats": (C.c_int64, [P, U64]),
            "orc_checkpoint_gather": (C.c_int64, [P, P, LaneS, LaneS, U64, P]),
            "orc_checkpoint_scatter": (C.c_int64, [P, P, LaneS, LaneS, U64, P]),
            "orc_payload_write": (C.c_int64, [P, I, P, P, P, P, P, P, P]),
            "orc_hadamard": (None, [P, I]),
            "orc_e2m1_rne": (F, [F]),
            "orc_fp4_scale_exp": (I, [F]),
            "orc_fp4_roundtrip": (None, [P, I]),
            "orc_indexer_qat": (None, [P, I]),
            "orc_index_score_heads": (F, [P, P, P, I, I]),
            "orc_indexer_topk_heads": (None, [P, P, P, P, P, I, P, P, C.c_int64]),
            "orc_payload_read": (C.c_int64, [P, I, P, P, P, P, P, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _weights(a, bf16: bool):
    """fp32 arrays pass as is; bf16 weights arrive as uint16 bit patterns."""
    if bf16:
        a = np.ascontiguousarray(a)
        assert a.dtype == np.uint16, "bf16 tensors are passed as uint16 bit patterns"
        return a
    return _f32(a)


# --------------------------------------------------------------------------
# Configuration and state
# --------------------------------------------------------------------------

@dataclass
class Layer:
    d_model: int
    head_dim: int
    n_rot: int
    idx_head_dim: int
    n_heads: int
    ratio: int
    swa: int
    top_k: int
    comp_cap: int
    idx_cap: int
    bf16: bool
    rms_eps: float
    attn_scale: float
    rope_base: float
    idx_heads: int = 0
    idx_qat: int = 0

    def c(self) -> Cfg:
        return Cfg(self.d_model, self.head_dim, self.n_rot, self.idx_head_dim, self.n_heads,
                   self.ratio, self.swa, self.top_k, self.comp_cap, self.idx_cap, int(self.bf16),
                   self.rms_eps, self.attn_scale, self.rope_base, self.idx_heads, self.idx_qat)

    @property
    def coff(self):
        return 2 if self.ratio == 4 else 1


class Lane:
    def __init__(self, cap: int, dl: int, coff: int, ratio: int):
        self.comp = np.full((max(cap, 1), dl), np.nan, dtype=np.float32)
        self.prequant = np.full((max(cap, 1), dl), np.nan, dtype=np.float32)
        rows = coff * ratio
        self.state_kv = np.zeros((max(rows, 1), coff * dl), dtype=np.float32)
        self.state_score = np.full((max(rows, 1), coff * dl), -np.inf, dtype=np.float32)

    def s(self) -> LaneS:
        return LaneS(self.comp.ctypes.data, self.state_kv.ctypes.data, self.state_score.ctypes.data,
                     self.prequant.ctypes.data)


class State:
    """One sequence's layer state, laid out as the pages' ds4_layer_cache."""

    def __init__(self, L: Layer):
        self.L = L
        self.raw = np.zeros((L.swa, L.head_dim), dtype=np.float32)
        self.attn = Lane(L.comp_cap, L.head_dim, L.coff, L.ratio)
        self.idx = Lane(L.idx_cap if L.ratio == 4 else 0, L.idx_head_dim, 2, 4 if L.ratio == 4 else 0)


# --------------------------------------------------------------------------
# Calls
# --------------------------------------------------------------------------

def num_threads() -> int:
    return lib().orc_num_threads()


def layer_ratio(variant: int, il: int) -> int:
    return lib().orc_layer_ratio(variant, il)


def raw_cap(ctx: int) -> int:
    return lib().orc_raw_cap(ctx)


def prefill_chunk(prompt_len: int, env_chunk: int = 0) -> int:
    return lib().orc_prefill_chunk(prompt_len, env_chunk)


def inv_freq(base: float, n_rot: int) -> np.ndarray:
    out = np.zeros(n_rot // 2, dtype=np.float32)
    lib().orc_inv_freq(base, n_rot, _p(out))
    return out


def project(W, h, bf16: bool = False) -> np.ndarray:
    W = _weights(W, bf16)
    h = _weights(h, bf16)
    T, K = h.shape
    N = W.shape[0]
    out = np.zeros((T, N), dtype=np.float32)
    lib().orc_project(_p(W), _p(h), int(bf16), T, K, N, _p(out))
    return out


def e4m3_rne(y) -> np.ndarray:
    y = _f32(y)
    f = lib().orc_e4m3_rne
    return np.array([f(float(v)) for v in y.ravel()], dtype=np.float32).reshape(y.shape)


def fp8_scale_exp(amax: float) -> int:
    return lib().orc_fp8_scale_exp(float(amax))


def fp8_roundtrip(rows, n_nope: int) -> np.ndarray:
    rows = _f32(rows).copy()
    flat = rows.reshape(-1, rows.shape[-1])
    for i in range(flat.shape[0]):
        r = np.ascontiguousarray(flat[i])
        lib().orc_fp8_roundtrip(_p(r), n_nope)
        flat[i] = r
    return flat.reshape(rows.shape)


def rope_tail(x, n_rot: int, p: int, inv_freq_table) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64).copy()
    f = _f32(inv_freq_table)
    lib().orc_rope_tail(_p(x), x.shape[-1], n_rot, p, _p(f))
    return x


def rmsnorm(x, gain=None, eps: float = 1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64).copy()
    g = None if gain is None else _f32(gain)
    lib().orc_rmsnorm(_p(x), x.shape[-1], _p(g), eps)
    return x


def compress_token(L: Layer, lane_is_attn: bool, ape, gain, lane: Lane, kv, score, pos: int):
    cfg = L.c()
    ape = _f32(ape)
    g = None if gain is None else _f32(gain)
    f = inv_freq(L.rope_base, L.n_rot)
    kv = _f32(kv)
    score = _f32(score)
    lib().orc_compress_token(C.byref(cfg), int(lane_is_attn), _p(ape), _p(g), _p(f), lane.s(),
                             _p(kv), _p(score), pos)


def state_init(st: State):
    cfg = st.L.c()
    st.raw[:] = 0.0
    if st.L.ratio != 0:
        lib().orc_state_init_lane(C.byref(cfg), 1, st.attn.s())
    if st.L.ratio == 4:
        lib().orc_state_init_lane(C.byref(cfg), 0, st.idx.s())


def compress(st: State, attn_w, idx_w, hidden, pos0: int):
    """A1-A8 over hidden [T, d_model]; attn_w/idx_w = (wkv, wgate, ape, norm)."""
    L = st.L
    if L.ratio == 0:
        return
    cfg = L.c()
    hidden = _weights(hidden, L.bf16)
    T = hidden.shape[0]
    keep = []

    def lw(w):
        wkv, wgate, ape, norm = w
        a = (_weights(wkv, L.bf16), _weights(wgate, L.bf16), _f32(ape), None if norm is None else _f32(norm))
        keep.append(a)
        return LaneW(a[0].ctypes.data, a[1].ctypes.data, a[2].ctypes.data,
                     None if a[3] is None else a[3].ctypes.data)

    aw = lw(attn_w)
    iw = lw(idx_w) if L.ratio == 4 else LaneW()
    buf = np.zeros(max(T, 1) * 2 * L.coff * max(L.head_dim, L.idx_head_dim), dtype=np.float32)
    lib().orc_compress(C.byref(cfg), C.byref(aw), C.byref(iw), st.attn.s(), st.idx.s(),
                       _p(hidden), T, pos0, _p(buf))


def index_score(q, row) -> float:
    q = _f32(q)
    row = _f32(row)
    return lib().orc_index_score(_p(q), _p(row), q.shape[0])


def topk(scores, visible: int, k: int) -> np.ndarray:
    s = _f32(scores)
    out = np.zeros(k, dtype=np.int32)
    lib().orc_topk(_p(s), visible, k, _p(out))
    return out


def indexer_topk(st: State, q_idx, positions, want_scores: bool = False):
    """Top-k lists [n, k] (and scores [n, max visible]) for queries at ``positions``."""
    L = st.L
    cfg = L.c()
    q_idx = _f32(q_idx)
    pos = np.ascontiguousarray(positions, dtype=np.uint64)
    n = pos.shape[0]
    out = np.zeros((n, L.top_k), dtype=np.int32)
    vmax = int((pos.max() + 1) // 4) if n else 0
    scores = np.full((n, max(vmax, 1)), np.nan, dtype=np.float32) if want_scores else None
    lib().orc_indexer_topk(C.byref(cfg), _p(st.idx.comp), _p(q_idx), _p(pos), n, _p(out),
                           _p(scores), max(vmax, 1))
    return (out, scores) if want_scores else out


def attention(st: State, q, raw_new, topk_lists, pos0: int) -> np.ndarray:
    """A11 for T queries at pos0.. (q [T, H, D], raw_new [T, D]); the ring is not changed."""
    L = st.L
    cfg = L.c()
    q = _f32(q)
    raw_new = _f32(raw_new)
    T = q.shape[0]
    tk = None if topk_lists is None else np.ascontiguousarray(topk_lists, dtype=np.int32)
    out = np.zeros((T, L.n_heads, L.head_dim), dtype=np.float32)
    lib().orc_attention(C.byref(cfg), _p(st.raw), _p(st.attn.comp), _p(q), _p(raw_new), _p(tk),
                        pos0, T, _p(out))
    return out


def ring_commit(st: State, raw_new, pos0: int):
    cfg = st.L.c()
    raw_new = _f32(raw_new)
    lib().orc_ring_commit(C.byref(cfg), _p(st.raw), _p(raw_new), pos0, raw_new.shape[0])


def checkpoint_floats(L: Layer, pos: int) -> int:
    cfg = L.c()
    return lib().orc_checkpoint_floats(C.byref(cfg), pos)


def checkpoint_scatter(st: State, pos: int, src: np.ndarray) -> None:
    """Restore `st` from a checkpoint body of `pos` tokens (in place)."""
    cfg = st.L.c()
    n = checkpoint_floats(st.L, pos)
    src = np.ascontiguousarray(src, dtype=np.float32)
    assert src.size >= n
    w = lib().orc_checkpoint_scatter(C.byref(cfg), _p(st.raw), st.attn.s(), st.idx.s(), pos, _p(src))
    assert w == n


def checkpoint_gather(st: State, pos: int) -> np.ndarray:
    cfg = st.L.c()
    n = checkpoint_floats(st.L, pos)
    dst = np.zeros(max(n, 1), dtype=np.float32)
    w = lib().orc_checkpoint_gather(C.byref(cfg), _p(st.raw), st.attn.s(), st.idx.s(), pos, _p(dst))
    assert w == n
    return dst[:n]


PAYLOAD_FIELDS = ("ctx_size", "prefill_chunk", "raw_cap", "raw_window", "comp_cap", "token_count", "layer_count",
                  "head_dim", "idx_head_dim", "vocab_size", "live_raw_rows")


def _stack_args(states):
    n = len(states)
    cfgs = (Cfg * n)(*[s.L.c() for s in states])
    rings = (C.c_void_p * n)(*[s.raw.ctypes.data for s in states])
    attn = (LaneS * n)(*[s.attn.s() for s in states])
    idx = (LaneS * n)(*[s.idx.s() for s in states])
    return cfgs, rings, attn, idx


def payload_size(states, fields) -> int:
    pos = fields[5]
    return 4 * (13 + fields[5] + fields[9] + 2 * len(states)) + 4 * sum(checkpoint_floats(s.L, pos) for s in states)


def payload_write(fields, states, tokens, logits) -> np.ndarray:
    """DSV4 payload bytes of the layer stack ``states`` (one State per layer, same sequence)."""
    f = np.ascontiguousarray(fields, dtype=np.uint32)
    assert f.size == 11
    tok = np.ascontiguousarray(tokens, dtype=np.uint32)
    lg = _f32(logits)
    assert tok.size == f[5] and lg.size == f[9]
    out = np.zeros(payload_size(states, [int(x) for x in f]), dtype=np.uint8)
    cfgs, rings, attn, idx = _stack_args(states)
    n = lib().orc_payload_write(_p(f), len(states), cfgs, rings, attn, idx, _p(tok) if tok.size else None,
                                _p(lg) if lg.size else None, _p(out))
    assert n == out.size
    return out


def payload_read(buf, states, max_tokens: int, vocab: int):
    """Restore ``states`` from payload bytes; returns (fields, tokens, logits)."""
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    n_tok = int(buf[28:32].view(np.uint32)[0])
    assert n_tok <= max_tokens and int(buf[44:48].view(np.uint32)[0]) == vocab, "payload larger than the buffers"
    f = np.zeros(11, dtype=np.uint32)
    tok = np.zeros(max(max_tokens, 1), dtype=np.uint32)
    lg = np.zeros(max(vocab, 1), dtype=np.float32)
    cfgs, rings, attn, idx = _stack_args(states)
    n = lib().orc_payload_read(_p(buf), len(states), cfgs, rings, attn, idx, _p(f), _p(tok), _p(lg))
    assert n >= 0, "payload magic or version mismatch"
    return f, tok[:f[5]], lg[:f[9]]


# --------------------------------------------------------------------------
# Full indexer: Hadamard + FP4 round trip, multi-head score
# --------------------------------------------------------------------------

def hadamard(x) -> np.ndarray:
    x = _f32(x).copy()
    flat = x.reshape(-1, x.shape[-1])
    for i in range(flat.shape[0]):
        r = np.ascontiguousarray(flat[i])
        lib().orc_hadamard(_p(r), r.shape[0])
        flat[i] = r
    return flat.reshape(x.shape)


def e2m1_rne(y) -> np.ndarray:
    y = _f32(y)
    f = lib().orc_e2m1_rne
    return np.array([f(float(v)) for v in y.ravel()], dtype=np.float32).reshape(y.shape)


def fp4_scale_exp(amax: float) -> int:
    return lib().orc_fp4_scale_exp(float(amax))


def fp4_roundtrip(x) -> np.ndarray:
    x = _f32(x).copy()
    flat = x.reshape(-1, x.shape[-1])
    for i in range(flat.shape[0]):
        r = np.ascontiguousarray(flat[i])
        lib().orc_fp4_roundtrip(_p(r), r.shape[0])
        flat[i] = r
    return flat.reshape(x.shape)


def indexer_qat(x) -> np.ndarray:
    x = _f32(x).copy()
    flat = x.reshape(-1, x.shape[-1])
    for i in range(flat.shape[0]):
        r = np.ascontiguousarray(flat[i])
        lib().orc_indexer_qat(_p(r), r.shape[0])
        flat[i] = r
    return flat.reshape(x.shape)


def index_score_heads(q, w, row) -> float:
    """q [heads][d] (after the round trip), w [heads], row [d]."""
    q, w, row = _f32(q), _f32(w), _f32(row)
    return lib().orc_index_score_heads(_p(q), _p(w), _p(row), q.shape[1], q.shape[0])


def indexer_topk_heads(st: State, q_raw, w, positions, want_scores: bool = False):
    """Multi-head top-k lists [n, k] (and scores) for queries q_raw [n, heads, d], weights w [n, heads]."""
    L = st.L
    cfg = L.c()
    q_raw, w = _f32(q_raw), _f32(w)
    assert q_raw.shape[1] == L.idx_heads and w.shape == q_raw.shape[:2]
    pos = np.ascontiguousarray(positions, dtype=np.uint64)
    n = pos.shape[0]
    out = np.zeros((n, L.top_k), dtype=np.int32)
    vmax = int((pos.max() + 1) // 4) if n else 0
    scores = np.full((n, max(vmax, 1)), np.nan, dtype=np.float32) if want_scores else None
    lib().orc_indexer_topk_heads(C.byref(cfg), _p(st.idx.comp), _p(q_raw), _p(w), _p(pos), n, _p(out), _p(scores),
                                 max(vmax, 1))
    return (out, scores) if want_scores else out
