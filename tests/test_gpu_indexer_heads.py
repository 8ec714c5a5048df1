"""The full indexer on the GPU (-m gpu): several indexer heads with per-query head
weights, and the Hadamard + FP4 round trip on the indexer rows and queries
("Metal グラフと圧縮 KV の実装を読む" §6 and §9).  The compressor's indexer rows are
checked as the FP8 rows are (the GPU's own pre-round-trip row re-quantised by the
oracle equals the GPU row bit for bit); scores and top-k lists are bit-exact against
the oracle on the GPU's own state, for prefill chunks and decode steps."""

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs, synth
from gpu_util import check_compress, device_layer, download, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    orc.build()


def _shape(heads, qat, d=128, dtype="bf16"):
    return configs.LayerShape(d_model=512, head_dim=128, n_rot=64, idx_head_dim=d, n_heads=8, ratio=4, top_k=64,
                              dtype=dtype, w_std=0.04, idx_heads=heads, idx_qat=qat)


def _queries(shape, seed, n, off):
    q = synth.normal(seed, 700, (n, shape.idx_heads, shape.idx_head_dim), offset=off * shape.idx_heads *
                     shape.idx_head_dim)
    w = synth.normal(seed, 701, (n, shape.idx_heads), offset=off * shape.idx_heads).abs() * 0.25
    return q, w


def _check_heads(st, q, w, positions, topk_gpu, scores_gpu, sample):
    for j in sample:
        tk, sc = orc.indexer_topk_heads(st, q[j:j + 1].numpy(), w[j:j + 1].numpy(), [positions[j]],
                                        want_scores=True)
        V = (positions[j] + 1) // 4
        np.testing.assert_array_equal(scores_gpu[j, :V], sc[0, :V], err_msg=f"scores query {j}")
        np.testing.assert_array_equal(topk_gpu[j], tk[0], err_msg=f"top-k query {j}")


@pytest.mark.parametrize("heads,qat,d", [(64, 1, 128), (4, 0, 128), (16, 1, 64)])
def test_indexer_heads_prefill_and_decode(heads, qat, d):
    shape = _shape(heads, qat, d)
    seed = 51 + heads + d
    dl, wa, wi = device_layer(shape, comp_cap=400, idx_cap=400, seed=seed, max_rows=512, with_prequant=True)
    report = {}
    pos = 0
    for n in (300, 437, 503):                       # ragged chunks; windows straddle the chunk ends
        h = configs.hidden(shape, seed, n, offset_tok=pos, device="cuda")
        before = download(dl)
        dl.compress_prefill(h, pos)
        after = download(dl)
        check_compress(before, after, wa, wi, h.cpu(), pos, report)
        pos += n
    st = download(dl)
    # prefill form: the next 200 queries of the sequence
    T = 200
    q, w = _queries(shape, seed, T, pos)
    V = (pos + T) // 4
    topk = torch.full((T, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((T, V), float("nan"), device="cuda")
    dl.indexer_topk_heads(q.cuda(), w.cuda(), [pos], 1, T, topk, scores, V)
    dl.sync()
    rng = np.random.default_rng(seed)
    sample = sorted(set([0, 1, T - 1] + rng.integers(0, T, 9).tolist()))
    _check_heads(st, q, w, [pos + j for j in range(T)], topk.cpu().numpy(), scores.cpu().numpy(), sample)
    # decode form: 6 sequences holding the same rows at staggered positions (some below 4: nothing visible)
    B = 6
    dd, _, _ = device_layer(shape, comp_cap=400, idx_cap=400, n_seq=B, seed=seed, max_rows=64)
    for b in range(B):
        dd.idx_comp[b] = dl.idx_comp[0]
    lens = [pos - 1, pos - 2, pos - 37, 515, 2, 255]
    q, w = _queries(shape, seed + 1, B, 0)
    vmax = max((p + 1) // 4 for p in lens)
    topk = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, vmax), float("nan"), device="cuda")
    dd.indexer_topk_heads(q.cuda(), w.cuda(), lens, B, 1, topk, scores, vmax)
    dd.sync()
    for b in range(B):
        _check_heads(st, q[b:b + 1], w[b:b + 1], [lens[b]], topk[b:b + 1].cpu().numpy(),
                     scores[b:b + 1].cpu().numpy(), [0])
    assert (topk[4] == -1).all()
