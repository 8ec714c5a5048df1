"""Seeded sweep of layer shapes against the oracle (-m gpu).

Each case draws one configuration from a fixed seed: ratio (0, 4, 128),
head_dim 64-512, indexer head_dim 64-256, RoPE width 4-128, head counts that
are multiples of 8 up to 128 (tensor-core and CUDA-core attention), ring sizes
32-256, top-k 1-2048, d_model not always a multiple of 64, bf16 or fp32
weights, the indexer lane's Hadamard + FP4 round trip on or off; then either a
prefill of one to three chunks of ragged lengths or a decode step of up to 33
sequences at staggered positions.  Every call is checked stage-wise on sampled
outputs, as in the parity tests: compressed rows and frontier, indexer scores
and lists (bit-exact), attention (tolerance), ring commit, checkpoint gather.
"""

import random

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs
from gpu_util import (check_attention_sampled, check_compress, check_indexer_sampled, device_layer, download,
                      require_gpu)
from test_gpu_parity import _gather_check, _run_chunk

pytestmark = pytest.mark.gpu

N_CASES = 40


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    orc.build()


def _draw(case: int):
    rng = random.Random(1000 + case)
    ratio = rng.choice([4, 4, 4, 128, 0])
    D = rng.choice([64, 128, 256, 512, 512])
    d = rng.choice([64, 128, 128, 256]) if ratio == 4 else 128
    rot_max = min(D, d if ratio == 4 else D, 128)
    n_rot = rng.choice([r for r in (4, 8, 32, 64, 128) if r <= rot_max])
    heads = rng.choice([h for h in (8, 16, 24, 40, 64, 64, 96, 128) if h * D <= 32768])
    shape = configs.LayerShape(d_model=rng.choice([256, 264, 512, 520, 1024]), head_dim=D, n_rot=n_rot,
                               idx_head_dim=d, n_heads=heads, ratio=ratio, swa=rng.choice([128, 128, 32, 64, 256]),
                               top_k=rng.choice([1, 8, 16, 100, 512, 512, 1000, 2048]),
                               dtype=rng.choice(["bf16", "bf16", "f32"]), w_std=0.04,
                               idx_qat=1 if (ratio == 4 and d in (64, 128) and rng.random() < 0.3) else 0)
    kind = rng.choice(["prefill", "prefill", "decode"])
    if kind == "prefill":
        plan = [rng.choice([1, 2, 3, 4, 5, 31, 64, 127, 128, 129, 257, 300, 513, 1100])
                for _ in range(rng.randint(1, 3))]
    else:
        B = rng.choice([1, 2, 5, 8, 17, 33])
        base = rng.choice([0, 3, 60, 127, 128, 200, 383, 700])
        plan = [base + rng.randint(0, 9) for _ in range(B)]
    return kind, shape, plan, rng.randint(0, 10 ** 6), rng


def _prefill(shape, Ts, seed, rng):
    total = sum(Ts)
    dl, wa, wi = device_layer(shape, comp_cap=total // max(shape.ratio, 1) + 2, idx_cap=total // 4 + 2, seed=seed,
                              gamma_std=0.1, max_rows=max(Ts))
    pos, report = 0, {}
    for T in Ts:
        sample = sorted(set([0, T - 1] + rng.sample(range(T), min(T, 4))))
        _run_chunk(dl, wa, wi, shape, seed, pos, T, report, sample=sample)
        pos += T
    _gather_check(dl, pos)


def _decode(shape, lens, seed, rng):
    B, ratio = len(lens), shape.ratio
    dl, wa, wi = device_layer(shape, comp_cap=max(lens) // max(ratio, 1) + 2, idx_cap=max(lens) // 4 + 2, n_seq=B,
                              seed=seed, max_rows=max(max(lens), B))
    for b in range(B):                                   # each sequence's state by its own prefill
        if lens[b] == 0:
            continue
        saved = dl.state
        dl.state = dl.seq_view(b)
        dl.compress_prefill(configs.hidden(shape, seed, lens[b], layer=b).cuda(), 0)
        dl.state = saved
        _, _, raw = configs.queries(shape, seed, lens[b], layer=b)
        for p in range(max(0, lens[b] - shape.swa), lens[b]):
            dl.raw[b, p % shape.swa] = raw[p].cuda()
    torch.cuda.synchronize()
    befores = [download(dl, b) for b in range(B)]
    hid = torch.stack([configs.hidden(shape, seed, 1, offset_tok=lens[b], layer=b)[0] for b in range(B)]).cuda()
    qs = [configs.queries(shape, seed, 1, offset_tok=lens[b], layer=b) for b in range(B)]
    q, q_idx, raw = (torch.cat([x[i] for x in qs]).cuda() for i in range(3))
    dl.compress_decode(hid, lens)
    topk = scores = None
    if ratio == 4:
        topk = torch.empty(B, shape.top_k, dtype=torch.int32, device="cuda")
        vmax = max(1, (max(lens) + 1) // 4)
        scores = torch.full((B, vmax), float("nan"), device="cuda")
        dl.indexer_topk(q_idx, lens, B, 1, topk, scores, vmax)
    out = torch.empty(B, shape.n_heads, shape.head_dim, device="cuda")
    torch.cuda.synchronize()
    after = [download(dl, b) for b in range(B)]
    dl.attention(q, raw, topk, lens, B, 1, out, commit_ring=True)
    dl.sync()
    for b in rng.sample(range(B), min(B, 4)):
        if ratio:
            check_compress(befores[b], after[b], wa, wi, hid[b:b + 1].cpu(), lens[b])
        if ratio == 4:
            check_indexer_sampled(after[b], q_idx[b:b + 1].cpu().numpy(), [lens[b]], topk[b:b + 1].cpu().numpy(),
                                  scores[b:b + 1].cpu().numpy(), [0])
        check_attention_sampled(after[b], q[b:b + 1].cpu().numpy(), raw[b:b + 1].cpu().numpy(),
                                None if topk is None else topk[b:b + 1].cpu().numpy(), out[b:b + 1].cpu().numpy(),
                                lens[b], [0])
        np.testing.assert_array_equal(dl.raw[b, lens[b] % shape.swa].cpu().numpy(), raw[b].cpu().numpy())


@pytest.mark.parametrize("case", range(N_CASES))
def test_shape_sweep(case):
    kind, shape, plan, seed, rng = _draw(case)
    if kind == "prefill":
        _prefill(shape, plan, seed, rng)
    else:
        _decode(shape, plan, seed, rng)
