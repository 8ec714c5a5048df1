"""Seeded synthetic inputs shared by the CUDA path, its tests and the oracle.

This module holds no arithmetic of the compressed-KV method: only a
counter-based random generator and the recipe that names one stream per
tensor.  Every tensor is a pure function of (seed, stream, element index), so
a chunk of a long input can be drawn on its own (``offset``) and equals the
matching slice of the whole tensor.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) evaluated at counter ``i`` of a per-tensor
key, two 53-bit uniforms per normal, Box-Muller transform in float64, rounded
to float32 (and from float32 to bfloat16 with round-to-nearest-even for bf16
tensors).  The arithmetic uses torch int64 tensors (two's-complement wrap
equals uint64 arithmetic) so the same code runs on the CPU and on a GPU.
Results on the two devices agree bit for bit in the integer part; the float64
log/cos of the transform may differ by an ulp between devices, so tests that
need identical bytes on both sides draw on the CPU and copy.
"""

from __future__ import annotations

import math

import torch

_MASK64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB


def _signed(x: int) -> int:
    x &= _MASK64
    return x - (1 << 64) if x >> 63 else x


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def _srl(z: torch.Tensor, k: int) -> torch.Tensor:
    """Logical right shift of int64 lanes viewed as uint64."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _signed(_M1)
    z = (z ^ _srl(z, 27)) * _signed(_M2)
    return z ^ _srl(z, 31)


def tensor_key(seed: int, stream: int) -> int:
    """64-bit key of one named tensor stream."""
    return _mix_int(_mix_int(seed) ^ (stream * _GOLDEN))


def uniform53(key: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """float64 uniforms in (0, 1] at counters start .. start+count-1."""
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    z = _mix(i * _signed(_GOLDEN) + _signed(key + _GOLDEN))
    return (_srl(z, 11).to(torch.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, stream: int, shape, std: float = 1.0, mean: float = 0.0,
           offset: int = 0, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """N(mean, std^2) samples of ``shape``; element e uses counters 2(offset+e), 2(offset+e)+1."""
    n = 1
    for s in shape:
        n *= int(s)
    key = tensor_key(seed, stream)
    u = uniform53(key, 2 * offset, 2 * n, device=device).view(n, 2)
    r = torch.sqrt(-2.0 * torch.log(u[:, 0]))
    x = r * torch.cos((2.0 * math.pi) * u[:, 1])
    x = (x * std + mean).to(torch.float32)
    if dtype == torch.bfloat16:
        x = x.to(torch.bfloat16)
    elif dtype != torch.float32:
        raise ValueError(f"unsupported dtype {dtype}")
    return x.view(*[int(s) for s in shape])


# Stream ids of the tensors of one layer; layer l uses stream 64*l + id.
STREAMS = {
    "attn.wkv": 1, "attn.wgate": 2, "attn.ape": 3, "attn.norm": 4,
    "idx.wkv": 5, "idx.wgate": 6, "idx.ape": 7, "idx.norm": 8,
    "hidden": 9, "q": 10, "q_idx": 11, "raw": 12,
}


def stream_id(name: str, layer: int = 0) -> int:
    return 64 * layer + STREAMS[name]
