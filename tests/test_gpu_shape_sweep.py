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
Two more sweeps draw the multi-head indexer (1 to 64 heads, QAT on or off;
scores and lists bit-exact) and the checkpoint restore (gather, scatter into a
fresh state, continue: bit for bit the uninterrupted run).
"""

import random

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs, synth
from gpu_util import (check_attention_sampled, check_compress, check_indexer_sampled, device_layer, download,
                      require_gpu)
from test_gpu_parity import _gather_check, _run_chunk

pytestmark = pytest.mark.gpu

N_CASES = 40
N_EXTRA = 12


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


@pytest.mark.parametrize("case", range(N_EXTRA))
def test_indexer_heads_sweep(case):
    kind, shape0, _, seed, rng = _draw(2000 + case)
    d = rng.choice([64, 128])
    heads = rng.choice([1, 2, 4, 8, 16, 33, 64])
    shape = configs.LayerShape(d_model=shape0.d_model, head_dim=shape0.head_dim, n_rot=min(shape0.n_rot, d),
                               idx_head_dim=d, n_heads=shape0.n_heads, ratio=4, swa=shape0.swa, top_k=shape0.top_k,
                               dtype=shape0.dtype, w_std=0.04, idx_heads=heads, idx_qat=rng.choice([0, 1]))
    Ts = [rng.choice([3, 64, 129, 300, 513]) for _ in range(rng.randint(1, 3))]
    T = rng.choice([1, 5, 64, 200])
    cap = (sum(Ts) + T) // 4 + 2
    dl, _, _ = device_layer(shape, comp_cap=cap, idx_cap=cap, seed=seed, max_rows=max(Ts + [T]))
    pos = 0
    for n in Ts:
        dl.compress_prefill(configs.hidden(shape, seed, n, offset_tok=pos, device="cuda"), pos)
        pos += n
    st = download(dl)
    q = synth.normal(seed, 700, (T, heads, d), offset=pos * heads * d)
    w = synth.normal(seed, 701, (T, heads), offset=pos * heads).abs() * 0.25
    V = max(1, (pos + T) // 4)
    topk = torch.full((T, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((T, V), float("nan"), device="cuda")
    dl.indexer_topk_heads(q.cuda(), w.cuda(), [pos], 1, T, topk, scores, V)
    dl.sync()
    tkg, scg = topk.cpu().numpy(), scores.cpu().numpy()
    for j in sorted(set([0, T - 1] + rng.sample(range(T), min(T, 4)))):
        tk, sc = orc.indexer_topk_heads(st, q[j:j + 1].numpy(), w[j:j + 1].numpy(), [pos + j], want_scores=True)
        Vj = (pos + j + 1) // 4
        np.testing.assert_array_equal(scg[j, :Vj], sc[0, :Vj], err_msg=f"scores query {j}")
        np.testing.assert_array_equal(tkg[j], tk[0], err_msg=f"top-k query {j}")


@pytest.mark.parametrize("case", range(N_EXTRA))
def test_restore_sweep(case):
    _, shape, _, seed, rng = _draw(3000 + case)
    T1, T2 = rng.choice([1, 5, 127, 301, 700]), rng.choice([1, 31, 170, 513])
    cap = (T1 + T2) // max(shape.ratio, 1) + 2
    icap = (T1 + T2) // 4 + 2
    dl, wa, wi = device_layer(shape, comp_cap=cap, idx_cap=icap, seed=seed, max_rows=max(T1, T2))
    _run_chunk(dl, wa, wi, shape, seed, 0, T1, {}, check=False)
    n = dl.checkpoint_floats(T1)
    body = torch.empty(n, device="cuda")
    dl.checkpoint_gather(0, T1, body)
    dl.sync()
    fresh, _, _ = device_layer(shape, comp_cap=cap, idx_cap=icap, seed=seed, max_rows=max(T1, T2))
    fresh.checkpoint_scatter(0, T1, body)
    fresh.sync()
    again = torch.empty(n, device="cuda")
    fresh.checkpoint_gather(0, T1, again)
    fresh.sync()
    assert torch.equal(again, body)
    tk_a, out_a = _run_chunk(dl, wa, wi, shape, seed, T1, T2, {}, check=False)
    tk_b, out_b = _run_chunk(fresh, wa, wi, shape, seed, T1, T2, {}, check=False)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    if tk_a is not None:
        assert torch.equal(tk_a, tk_b)
