"""Shared test helpers: input conversion and an independent window-form restatement
of the compressor used to pin the oracle's token-recurrent implementation."""

from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from compressed_kv_sparse_compressor_gb300 import configs


def np_in(t: torch.Tensor) -> np.ndarray:
    """Host numpy view of a generated tensor; bf16 becomes its uint16 bit pattern."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def np_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def orc_layer(shape: configs.LayerShape, comp_cap: int, idx_cap: int = 0) -> oracle.Layer:
    return oracle.Layer(d_model=shape.d_model, head_dim=shape.head_dim, n_rot=shape.n_rot,
                        idx_head_dim=shape.idx_head_dim, n_heads=shape.n_heads, ratio=shape.ratio,
                        swa=shape.swa, top_k=shape.top_k, comp_cap=comp_cap, idx_cap=idx_cap,
                        bf16=(shape.dtype == "bf16"), rms_eps=shape.rms_eps,
                        attn_scale=shape.attn_scale, rope_base=shape.rope_base, idx_heads=shape.idx_heads,
                        idx_qat=shape.idx_qat)


def lane_np(w):
    wkv, wgate, ape, norm = w
    return (np_in(wkv), np_in(wgate), np_in(ape), np_in(norm))


# ---------------------------------------------------------------------------
# Independent restatement (window form, numpy float64 + torch's float8 cast).
# It forms each compressed row directly from the tokens of its window instead
# of replaying the frontier's store / pool / shift recurrence.
# ---------------------------------------------------------------------------

def e4m3_torch(y: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32))
    t = torch.clamp(t, -448.0, 448.0)
    return t.to(torch.float8_e4m3fn).to(torch.float32).numpy()


def fp8_block_exp(amax: float) -> int:
    if amax == 0.0:
        return 0
    m, E = math.frexp(amax)        # amax = m * 2^E, m in [0.5, 1)
    for e in range(E - 12, E + 2):
        if amax <= 448.0 * 2.0 ** e:
            return e
    raise AssertionError


def fp8_rows_window_form(rows: np.ndarray, n_nope: int) -> np.ndarray:
    out = np.array(rows, dtype=np.float32, copy=True)
    for r in out:
        for b0 in range(0, n_nope, 64):
            blk = r[b0:min(b0 + 64, n_nope)]
            e = fp8_block_exp(float(np.max(np.abs(blk))) if blk.size else 0.0)
            y = (blk.astype(np.float64) * 2.0 ** -e).astype(np.float32)
            r[b0:b0 + blk.size] = (e4m3_torch(y).astype(np.float64) * 2.0 ** e).astype(np.float32)
    return out


def window_form_lane(shape: configs.LayerShape, w, hidden: torch.Tensor, lane_is_attn: bool):
    """Compressed rows (pre-FP8 and final) of one lane for tokens 0..T-1."""
    wkv, wgate, ape, gain = (np_f64(x) for x in w)
    h = np_f64(hidden)
    r = shape.ratio
    dl = shape.head_dim if lane_is_attn else shape.idx_head_dim
    kv = (h @ wkv.T).astype(np.float32)
    sc = (h @ wgate.T).astype(np.float32)
    T = h.shape[0]
    sa = np.stack([(sc[t] + ape[t % r].astype(np.float32)).astype(np.float32) for t in range(T)])
    inv = np.array([np.float32(shape.rope_base ** (-2.0 * i / shape.n_rot)) for i in range(shape.n_rot // 2)],
                   dtype=np.float32)
    pre = []
    for c in range(T // r):
        if r == 4:
            toks_prev = [(c - 1) * 4 + q for q in range(4)]
            toks_cur = [c * 4 + q for q in range(4)]
            ck = [kv[t, :dl] if t >= 0 else np.zeros(dl, np.float32) for t in toks_prev] + \
                 [kv[t, dl:] for t in toks_cur]
            cs = [sa[t, :dl] if t >= 0 else np.full(dl, -np.inf, np.float32) for t in toks_prev] + \
                 [sa[t, dl:] for t in toks_cur]
        else:
            ck = [kv[t] for t in range(c * r, (c + 1) * r)]
            cs = [sa[t] for t in range(c * r, (c + 1) * r)]
        ck = np.stack(ck).astype(np.float64)
        cs = np.stack(cs).astype(np.float64)
        wts = np.exp(cs - cs.max(axis=0, keepdims=True))
        pooled = (wts * ck).sum(0) / wts.sum(0)
        x = pooled / np.sqrt(np.mean(pooled ** 2) + shape.rms_eps) * gain
        tail = x[dl - shape.n_rot:]
        z = tail[0::2] + 1j * tail[1::2]
        ang = (np.float32(c * r) * inv).astype(np.float32).astype(np.float64)
        z = z * np.exp(1j * ang)
        x = x.copy()
        x[dl - shape.n_rot::2] = z.real
        x[dl - shape.n_rot + 1::2] = z.imag
        pre.append(x.astype(np.float32))
    pre = np.stack(pre) if pre else np.zeros((0, dl), np.float32)
    fin = fp8_rows_window_form(pre, dl - shape.n_rot) if lane_is_attn else pre.copy()
    return pre, fin, kv, sa


def dense_attention(q, rows_list, scale):
    """softmax(q x^T * scale) x for one query over an explicit row matrix (float64)."""
    X = np.asarray(rows_list, dtype=np.float64)
    Q = np.asarray(q, dtype=np.float64)
    L = Q @ X.T * scale
    L = L - L.max(axis=-1, keepdims=True)
    P = np.exp(L)
    P = P / P.sum(axis=-1, keepdims=True)
    return P @ X
