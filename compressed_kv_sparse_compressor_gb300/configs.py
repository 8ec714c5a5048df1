"""The five synthetic workloads of the compressed-KV attention path.

Shapes follow the DeepSeek-V4 Flash figures quoted in "Metal グラフと圧縮 KV の実装を読む"
(§2 raw ring of 128 rows, §3 4096-token prefill chunks, §6 indexer head_dim 128 and
top-k 512, §8 head_dim 512 with a 64-dim RoPE tail).  Values the pages leave open
(weight scales, APE scale, seeds) are the workload's own choices.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

from . import synth


@dataclass(frozen=True)
class LayerShape:
    d_model: int
    head_dim: int          # D: attention row width (K = V = the stored row)
    n_rot: int             # R: RoPE tail width
    idx_head_dim: int      # d: indexer row width (ratio-4 layers)
    n_heads: int           # H: query heads sharing the single KV row
    ratio: int             # 0 (uncompressed), 4 or 128
    swa: int = 128         # raw sliding-window ring rows
    top_k: int = 512
    dtype: str = "bf16"    # weights and hidden states: "f32" or "bf16"
    w_std: float = 0.02
    ape_std: float = 0.1
    rope_base: float = 10000.0
    rms_eps: float = 1e-6
    idx_heads: int = 0     # indexer query heads of the multi-head score (0: one query vector)
    idx_qat: int = 0       # 1: the indexer rows and queries take the Hadamard + FP4 round trip

    @property
    def coff(self) -> int:
        return 2 if self.ratio == 4 else 1

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def attn_scale(self) -> float:
        return float(torch.tensor(1.0 / self.head_dim ** 0.5, dtype=torch.float32))


@dataclass(frozen=True)
class Workload:
    name: str
    layer: LayerShape
    ratios: tuple = ()          # per-layer ratios of a stack (empty: one layer)
    n_tok: int = 0              # prefill tokens per sequence
    chunk: int = 4096
    n_seq: int = 1
    ctx: int = 0                # decode: context already in the state
    seed: int = 0
    note: str = ""
    extra: dict = field(default_factory=dict)

    def layers(self):
        if not self.ratios:
            return [self.layer]
        return [replace(self.layer, ratio=r) for r in self.ratios]


C1 = Workload(
    name="c1_ratio4_T64_f32",
    layer=LayerShape(d_model=256, head_dim=128, n_rot=64, idx_head_dim=64, n_heads=8,
                     ratio=4, top_k=8, dtype="f32", w_std=1.0 / 16.0),
    n_tok=64, chunk=64, seed=0,
    note="one ratio-4 layer, 64-token prefill, fp32 throughout")

C2 = Workload(
    name="c2_ratio128_T8192_bf16",
    layer=LayerShape(d_model=4096, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64,
                     ratio=128),
    n_tok=8192, chunk=4096, seed=2,
    note="one ratio-128 layer, 8192-token prefill in two 4096-token chunks")

C3 = Workload(
    name="c3_flash8_T32768_bf16",
    layer=LayerShape(d_model=4096, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64,
                     ratio=4),
    ratios=(0, 0, 4, 128, 4, 128, 4, 128),
    n_tok=32768, chunk=4096, seed=3,
    note="Flash-style 8-layer stack, 32768-token prefill in 4096-token chunks")

C4 = Workload(
    name="c4_decode_B32_ctx65536_bf16",
    layer=LayerShape(d_model=4096, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64,
                     ratio=4),
    n_seq=32, ctx=65536, seed=4,
    note="decode step, 32 sequences at 65536 + (b mod 4) context, ratio-4 layer")

C5 = Workload(
    name="c5_ratio4_T131072_bf16",
    layer=LayerShape(d_model=4096, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64,
                     ratio=4),
    n_tok=131072, chunk=4096, seed=5,
    note="long-context ratio-4 layer, 131072-token prefill, then checkpoint gather")

ALL = {w.name: w for w in (C1, C2, C3, C4, C5)}

# The Pro variant's layer table ("Metal グラフと圧縮 KV の実装を読む" §1: layers 0-1 at
# ratio 128 instead of uncompressed, then even layers ratio 4, odd layers ratio 128) on
# the same layer shapes as the Flash stack, 8192 tokens per layer in two chunks.
PRO = Workload(
    name="pro8_T8192_bf16",
    layer=LayerShape(d_model=4096, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64,
                     ratio=4),
    ratios=(128, 128, 4, 128, 4, 128, 4, 128),
    n_tok=8192, chunk=4096, seed=6,
    note="Pro-style 8-layer stack, 8192-token prefill in 4096-token chunks")


def comp_caps(shape: LayerShape, max_tokens: int):
    """Rows the compressed arrays must hold after ``max_tokens`` tokens."""
    if shape.ratio == 0:
        return 0, 0
    attn = max_tokens // shape.ratio
    idx = max_tokens // 4 if shape.ratio == 4 else 0
    return attn, idx


# ---------------------------------------------------------------------------
# Tensor recipes.  Each returns host (or device) tensors drawn from the seeded
# generator; nothing here computes any part of the method.
# ---------------------------------------------------------------------------

def lane_weights(shape: LayerShape, seed: int, layer: int, lane: str, device="cpu",
                 gamma_std: float = 0.0):
    """wkv, wgate [coff*Dl, d_model]; ape [ratio, coff*Dl]; norm gamma [Dl] (ones unless gamma_std>0)."""
    dl = shape.head_dim if lane == "attn" else shape.idx_head_dim
    width = shape.coff * dl
    dt = shape.torch_dtype
    wkv = synth.normal(seed, synth.stream_id(f"{lane}.wkv", layer), (width, shape.d_model),
                       std=shape.w_std, device=device, dtype=dt)
    wgate = synth.normal(seed, synth.stream_id(f"{lane}.wgate", layer), (width, shape.d_model),
                         std=shape.w_std, device=device, dtype=dt)
    ape = synth.normal(seed, synth.stream_id(f"{lane}.ape", layer), (shape.ratio, width),
                       std=shape.ape_std, device=device)
    if gamma_std > 0.0:
        norm = synth.normal(seed, synth.stream_id(f"{lane}.norm", layer), (dl,),
                            std=gamma_std, mean=1.0, device=device)
    else:
        norm = torch.ones(dl, dtype=torch.float32, device=device)
    return wkv, wgate, ape, norm


def hidden(shape: LayerShape, seed: int, n_tok: int, offset_tok: int = 0, device="cpu", layer: int = 0):
    return synth.normal(seed, synth.stream_id("hidden", layer), (n_tok, shape.d_model),
                        offset=offset_tok * shape.d_model, device=device, dtype=shape.torch_dtype)


def queries(shape: LayerShape, seed: int, n_tok: int, offset_tok: int = 0, device="cpu", layer: int = 0):
    """q [n, H, D] (already rotated by the caller), q_idx [n, d], raw rows [n, D]; all fp32 N(0,1)."""
    q = synth.normal(seed, synth.stream_id("q", layer), (n_tok, shape.n_heads, shape.head_dim),
                     offset=offset_tok * shape.n_heads * shape.head_dim, device=device)
    q_idx = synth.normal(seed, synth.stream_id("q_idx", layer), (n_tok, shape.idx_head_dim),
                         offset=offset_tok * shape.idx_head_dim, device=device)
    raw = synth.normal(seed, synth.stream_id("raw", layer), (n_tok, shape.head_dim),
                       offset=offset_tok * shape.head_dim, device=device)
    return q, q_idx, raw
