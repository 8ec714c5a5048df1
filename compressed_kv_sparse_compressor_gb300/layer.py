"""Device-side layer object over the C ABI: owns the torch tensors that back one
layer's weights, state and workspace, builds the ABI structs and calls the
ABI.  Marshalling only; torch provides device memory and the stream."""

from __future__ import annotations

import ctypes as C

import torch

from . import abi
from .configs import LayerShape


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream():
    return torch.cuda.current_stream().cuda_stream


class DeviceLayer:
    def __init__(self, shape: LayerShape, comp_cap: int, idx_cap: int = 0, n_seq: int = 1, max_rows: int = 4096,
                 device="cuda", with_prequant: bool = False):
        self.shape = shape
        self.n_seq = n_seq
        self.device = device
        r = shape.ratio
        coff = shape.coff
        D, d = shape.head_dim, shape.idx_head_dim
        self.comp_cap = max(comp_cap, 1) if r else 0
        self.idx_cap = max(idx_cap, 1) if r == 4 else 0
        self.cfg = abi.LayerCfg(
            d_model=shape.d_model, head_dim=D, n_rot=shape.n_rot, idx_head_dim=d, n_heads=shape.n_heads,
            ratio=r, swa=shape.swa, top_k=shape.top_k, comp_cap=self.comp_cap, idx_cap=self.idx_cap,
            dtype=abi.DS4C_F32 if shape.dtype == "f32" else abi.DS4C_BF16, rms_eps=shape.rms_eps,
            attn_scale=shape.attn_scale, rope_base=shape.rope_base, idx_heads=shape.idx_heads,
            idx_qat=shape.idx_qat)
        f32 = dict(dtype=torch.float32, device=device)
        self.raw = torch.zeros(n_seq, shape.swa, D, **f32)
        self.attn_comp = self.attn_kv = self.attn_score = self.attn_pre = self.attn_split = None
        self.idx_comp = self.idx_kv = self.idx_score = None
        if r:
            self.attn_comp = torch.zeros(n_seq, self.comp_cap, D, **f32)
            self.attn_kv = torch.zeros(n_seq, coff * r, coff * D, **f32)
            self.attn_score = torch.zeros(n_seq, coff * r, coff * D, **f32)
            if with_prequant:
                self.attn_pre = torch.zeros(n_seq, self.comp_cap, D, **f32)
            if abi.ds4c_attn_uses_tensor_cores(self.cfg):
                # bf16 hi / lo mirror of the compressed rows, read by the tensor-core attention
                self.attn_split = torch.zeros(n_seq, self.comp_cap, 2, D, dtype=torch.int16, device=device)
        self.idx_pre = None
        if r == 4:
            self.idx_comp = torch.zeros(n_seq, self.idx_cap, d, **f32)
            if with_prequant:
                self.idx_pre = torch.zeros(n_seq, self.idx_cap, d, **f32)
            self.idx_kv = torch.zeros(n_seq, 8, 2 * d, **f32)
            self.idx_score = torch.zeros(n_seq, 8, 2 * d, **f32)
        self.state = abi.LayerState(
            raw=_ptr(self.raw),
            attn=abi.LaneState(_ptr(self.attn_comp), _ptr(self.attn_kv), _ptr(self.attn_score), _ptr(self.attn_pre),
                               _ptr(self.attn_split)),
            idx=abi.LaneState(_ptr(self.idx_comp), _ptr(self.idx_kv), _ptr(self.idx_score), _ptr(self.idx_pre), None))
        self.ws_bytes = abi.ds4c_workspace_bytes(self.cfg, max_rows, n_seq)
        if self.ws_bytes == 0:
            raise abi.Ds4cError(abi.DS4C_ERR_SHAPE, "ds4c_workspace_bytes")
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        self.attn_w = self.idx_w = None
        self._keep = []

    # -- weights -------------------------------------------------------------
    def set_weights(self, attn, idx=None):
        """attn / idx = (wkv, wgate, ape, norm) tensors (moved to the device)."""
        def lw(w):
            t = [None if x is None else x.to(self.device).contiguous() for x in w]
            self._keep.append(t)
            return abi.LaneWeights(_ptr(t[0]), _ptr(t[1]), _ptr(t[2]), _ptr(t[3]))
        if self.shape.ratio:
            self.attn_w = lw(attn)
        if self.shape.ratio == 4:
            self.idx_w = lw(idx)

    # -- calls -----------------------------------------------------------------
    def state_init(self):
        abi.check(abi.ds4c_state_init(self.cfg, self.state, self.n_seq, _stream()), "ds4c_state_init")

    def compress_prefill(self, hidden: torch.Tensor, pos0: int):
        abi.check(abi.ds4c_compress_prefill(self.cfg, self.attn_w, self.idx_w, self.state, _ptr(hidden),
                                            hidden.shape[0], pos0, _ptr(self.ws), self.ws_bytes, _stream()),
                  "ds4c_compress_prefill")

    def compress_prefill_timed(self, hidden: torch.Tensor, pos0: int, after_projection: torch.cuda.Event):
        """ds4c_compress_prefill with `after_projection` recorded between the projection GEMM and the
        fused compressor (a measurement hook)."""
        after_projection.record()       # creates the event on this device; the library re-records it in the call
        abi.check(abi.ds4c_compress_prefill_timed(self.cfg, self.attn_w, self.idx_w, self.state, _ptr(hidden),
                                                  hidden.shape[0], pos0, _ptr(self.ws), self.ws_bytes,
                                                  after_projection.cuda_event, _stream()),
                  "ds4c_compress_prefill_timed")

    def compress_decode(self, hidden: torch.Tensor, positions):
        pos = abi.u64_array(positions)
        abi.check(abi.ds4c_compress_decode_step(self.cfg, self.attn_w, self.idx_w, self.state, _ptr(hidden), pos,
                                                len(positions), _ptr(self.ws), self.ws_bytes, _stream()),
                  "ds4c_compress_decode_step")

    def indexer_topk(self, q_idx, positions, n_seq, n_tok, topk, scores=None, score_stride=0):
        pos = abi.u64_array(positions)
        abi.check(abi.ds4c_indexer_topk(self.cfg, self.state, _ptr(q_idx), pos, n_seq, n_tok, _ptr(topk),
                                        _ptr(scores), score_stride, _ptr(self.ws), self.ws_bytes, _stream()),
                  "ds4c_indexer_topk")

    def indexer_topk_heads(self, q_idx, w_idx, positions, n_seq, n_tok, topk, scores=None, score_stride=0):
        pos = abi.u64_array(positions)
        abi.check(abi.ds4c_indexer_topk_heads(self.cfg, self.state, _ptr(q_idx), _ptr(w_idx), pos, n_seq, n_tok,
                                              _ptr(topk), _ptr(scores), score_stride, _ptr(self.ws), self.ws_bytes,
                                              _stream()), "ds4c_indexer_topk_heads")

    def attention(self, q, raw_new, topk, positions, n_seq, n_tok, out, commit_ring=True):
        pos = abi.u64_array(positions)
        abi.check(abi.ds4c_sparse_swa_attn(self.cfg, self.state, _ptr(q), _ptr(raw_new), _ptr(topk), pos, n_seq,
                                           n_tok, _ptr(out), commit_ring, _ptr(self.ws), self.ws_bytes, _stream()),
                  "ds4c_sparse_swa_attn")

    def checkpoint_floats(self, pos: int) -> int:
        return abi.ds4c_checkpoint_floats(self.cfg, pos)

    def checkpoint_gather(self, seq: int, pos: int, dst: torch.Tensor) -> int:
        written = C.c_size_t(0)
        abi.check(abi.ds4c_checkpoint_gather(self.cfg, self.state, seq, pos, _ptr(dst), dst.numel(),
                                             C.byref(written), _stream()), "ds4c_checkpoint_gather")
        return written.value

    def checkpoint_scatter(self, seq: int, pos: int, src: torch.Tensor) -> None:
        abi.check(abi.ds4c_checkpoint_scatter(self.cfg, self.state, seq, pos, _ptr(src), src.numel(), _stream()),
                  "ds4c_checkpoint_scatter")

    def sync(self):
        abi.check(abi.ds4c_sync_status(_stream()), "ds4c_sync_status")

    # -- per-sequence views ------------------------------------------------------
    def seq_view(self, b: int):
        """A state struct that addresses sequence b only (for n_seq == 1 calls)."""
        def off(t):
            return None if t is None else t[b].data_ptr()
        return abi.LayerState(
            raw=off(self.raw),
            attn=abi.LaneState(off(self.attn_comp), off(self.attn_kv), off(self.attn_score), off(self.attn_pre),
                               off(self.attn_split)),
            idx=abi.LaneState(off(self.idx_comp), off(self.idx_kv), off(self.idx_score), off(self.idx_pre), None))
