"""Full-size workloads on the GPU, checked on sampled outputs (-m gpu).

The GPU runs each workload in full, with the chunking the benchmark uses; the
oracle recomputes stage-wise one chunk (or one decode step) from the GPU's own
state before it, plus sampled indexer and attention queries, and the whole
checkpoint gather bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs
from gpu_util import (ATOL, RTOL, check_attention_sampled, check_compress, check_indexer_sampled, check_split_mirror,
                      device_layer, download, require_gpu, unexplained_fp8_flips)
from helpers import lane_np, np_in, orc_layer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    orc.build()


def _chunk(dl, shape, seed, p0, n, layer=0, topk=None, out=None):
    dev = "cuda"
    h = configs.hidden(shape, seed, n, offset_tok=p0, device=dev, layer=layer)
    q, q_idx, raw = configs.queries(shape, seed, n, offset_tok=p0, device=dev, layer=layer)
    dl.compress_prefill(h, p0)
    tk = None
    if shape.ratio == 4:
        tk = torch.empty(n, shape.top_k, dtype=torch.int32, device=dev) if topk is None else topk
        dl.indexer_topk(q_idx, [p0], 1, n, tk)
    o = torch.empty(n, shape.n_heads, shape.head_dim, device=dev) if out is None else out
    dl.attention(q, raw, tk, [p0], 1, n, o, commit_ring=True)
    return h, q, q_idx, raw, tk, o


def _checked_chunk(dl, wa, wi, shape, seed, p0, n, sample, layer=0):
    dev = "cuda"
    h = configs.hidden(shape, seed, n, offset_tok=p0, device=dev, layer=layer)
    q, q_idx, raw = configs.queries(shape, seed, n, offset_tok=p0, device=dev, layer=layer)
    before = download(dl)
    dl.compress_prefill(h, p0)
    after = download(dl)
    if shape.ratio:
        check_compress(before, after, wa, wi, h.cpu(), p0)
        check_split_mirror(dl)
    tk = None
    if shape.ratio == 4:
        vis = (p0 + n) // 4
        tk = torch.empty(n, shape.top_k, dtype=torch.int32, device=dev)
        sc = torch.empty(n, vis, device=dev)
        dl.indexer_topk(q_idx, [p0], 1, n, tk, sc, vis)
        torch.cuda.synchronize()
        rows = np.asarray(sample)
        check_indexer_sampled(after, q_idx[rows].cpu().numpy(), [p0 + j for j in sample], tk[rows].cpu().numpy(),
                              sc[rows].cpu().numpy(), range(len(sample)))
    out = torch.empty(n, shape.n_heads, shape.head_dim, device=dev)
    dl.attention(q, raw, tk, [p0], 1, n, out, commit_ring=True)
    dl.sync()
    check_attention_sampled(after, q.cpu().numpy(), raw.cpu().numpy(), None if tk is None else tk.cpu().numpy(),
                            out.cpu().numpy(), p0, sample)


def _gather_check(dl, pos):
    n = dl.checkpoint_floats(pos)
    dst = torch.empty(n, device="cuda")
    assert dl.checkpoint_gather(0, pos, dst) == n
    dl.sync()
    np.testing.assert_array_equal(dst.cpu().numpy(), orc.checkpoint_gather(download(dl), pos))


def _check_windows_across_the_run(dl, wa, wi, shape, seed, windows):
    """Compressed rows of windows sampled over the whole prefill, both lanes, against the
    oracle: row c of a ratio-4 lane depends only on tokens 4(c-1) .. 4c+3, so the oracle
    compresses those eight tokens from a fresh state and takes its window c."""
    st = download(dl)
    n_nope = shape.head_dim - shape.n_rot
    attn_w, idx_w = lane_np(wa), lane_np(wi)
    gp, gc, op, oc = [], [], [], []
    for c in windows:
        p0 = max(0, 4 * (c - 1))
        h = configs.hidden(shape, seed, 4 * c + 4 - p0, offset_tok=p0)
        ref = orc.State(orc_layer(shape, c + 1, c + 1))
        orc.state_init(ref)
        orc.compress(ref, attn_w, idx_w, np_in(h), p0)
        np.testing.assert_allclose(st.attn.prequant[c], ref.attn.prequant[c], rtol=RTOL, atol=ATOL,
                                   err_msg=f"attn pre-FP8 row {c}")
        np.testing.assert_array_equal(orc.fp8_roundtrip(st.attn.prequant[c:c + 1], n_nope)[0], st.attn.comp[c],
                                      err_msg=f"attn FP8 arithmetic row {c}")
        np.testing.assert_allclose(st.attn.comp[c, n_nope:], ref.attn.comp[c, n_nope:], rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(st.idx.comp[c], ref.idx.comp[c], rtol=RTOL, atol=ATOL, err_msg=f"idx row {c}")
        gp.append(st.attn.prequant[c]); gc.append(st.attn.comp[c]); op.append(ref.attn.prequant[c])
        oc.append(ref.attn.comp[c])
    assert unexplained_fp8_flips(np.array(gp), np.array(gc), np.array(op), np.array(oc), n_nope) == 0


def test_c5_full():
    """Long-context ratio-4 layer: 131072 tokens in 32 chunks, then the gather."""
    w = configs.C5
    shape = w.layer
    T, C = w.n_tok, w.chunk
    dl, wa, wi = device_layer(shape, comp_cap=T // 4, idx_cap=T // 4, seed=w.seed, max_rows=C, with_prequant=True)
    topk = torch.empty(C, shape.top_k, dtype=torch.int32, device="cuda")
    out = torch.empty(C, shape.n_heads, shape.head_dim, device="cuda")
    for c in range(T // C - 1):
        _chunk(dl, shape, w.seed, c * C, C, topk=topk, out=out)
    dl.sync()
    rng = np.random.default_rng(5)
    sample = sorted(set([0, 1, 2, 3, C - 1] + rng.integers(0, C, 11).tolist()))
    _checked_chunk(dl, wa, wi, shape, w.seed, T - C, C, sample)
    _gather_check(dl, T)
    # 64 windows over all 32 chunks: the first, chunk edges (the last window of a chunk and the
    # first of the next), the last, and random ones
    n_win = T // 4
    edges = [c for k in (1, 7, 15, 16, 31) for c in (k * (C // 4) - 1, k * (C // 4))]
    windows = set([0, 1, n_win - 1] + edges)
    while len(windows) < 64:
        windows.add(int(rng.integers(0, n_win)))
    windows = sorted(windows)
    _check_windows_across_the_run(dl, wa, wi, shape, w.seed, windows)


def test_c4_decode_full():
    """32 sequences at 65536 + (b mod 4): state built by the compressor, one decode step."""
    w = configs.C4
    shape = w.layer
    B = w.n_seq
    lens = [w.ctx + (b % 4) for b in range(B)]
    cap = (max(lens) + 1) // 4 + 1
    dl, wa, wi = device_layer(shape, comp_cap=cap, idx_cap=cap, n_seq=B, seed=w.seed, max_rows=4096)
    saved = dl.state
    for b in range(B):
        dl.state = dl.seq_view(b)
        for p0 in range(0, lens[b], 4096):
            n = min(4096, lens[b] - p0)
            dl.compress_prefill(configs.hidden(shape, w.seed, n, offset_tok=p0, device="cuda", layer=b), p0)
        dl.state = saved
        _, _, raw = configs.queries(shape, w.seed, shape.swa, offset_tok=lens[b] - shape.swa, device="cuda", layer=b)
        for i, p in enumerate(range(lens[b] - shape.swa, lens[b])):
            dl.raw[b, p % shape.swa] = raw[i]
    dl.sync()
    befores = [download(dl, b) for b in range(B)]
    hid = torch.cat([configs.hidden(shape, w.seed, 1, offset_tok=lens[b], device="cuda", layer=b) for b in range(B)])
    qs = [configs.queries(shape, w.seed, 1, offset_tok=lens[b], device="cuda", layer=b) for b in range(B)]
    q = torch.cat([x[0] for x in qs])
    q_idx = torch.cat([x[1] for x in qs])
    raw = torch.cat([x[2] for x in qs])
    dl.compress_decode(hid, lens)
    vmax = (max(lens) + 1) // 4
    topk = torch.empty(B, shape.top_k, dtype=torch.int32, device="cuda")
    scores = torch.empty(B, vmax, device="cuda")
    dl.indexer_topk(q_idx, lens, B, 1, topk, scores, vmax)
    dl.sync()
    afters = [download(dl, b) for b in range(B)]
    out = torch.empty(B, shape.n_heads, shape.head_dim, device="cuda")
    dl.attention(q, raw, topk, lens, B, 1, out, commit_ring=True)
    dl.sync()
    emitted = 0
    for b in range(B):
        check_compress(befores[b], afters[b], wa, wi, hid[b:b + 1].cpu(), lens[b])
        emitted += (lens[b] + 1) % 4 == 0
        check_indexer_sampled(afters[b], q_idx[b:b + 1].cpu().numpy(), [lens[b]], topk[b:b + 1].cpu().numpy(),
                              scores[b:b + 1].cpu().numpy(), [0])
        check_attention_sampled(afters[b], q[b:b + 1].cpu().numpy(), raw[b:b + 1].cpu().numpy(),
                                topk[b:b + 1].cpu().numpy(), out[b:b + 1].cpu().numpy(), lens[b], [0])
    assert emitted == B // 4


def test_c3_stack():
    """Flash-style 8-layer stack, 32768 tokens per layer; the last chunk of one
    layer of each ratio (0, 4, 128) is checked stage-wise, every layer runs."""
    w = configs.C3
    T, C = w.n_tok, w.chunk
    checked = {0: False, 4: False, 128: False}
    rng = np.random.default_rng(3)
    for li, shape in enumerate(w.layers()):
        r = shape.ratio
        dl, wa, wi = device_layer(shape, comp_cap=max(T // max(r, 1), 1), idx_cap=T // 4 if r == 4 else 0,
                                  seed=w.seed, layer=li, max_rows=C, with_prequant=True)
        check = not checked[r]
        last = T // C - 1 if check else T // C
        for c in range(last):
            _chunk(dl, shape, w.seed, c * C, C, layer=li)
        if check:
            dl.sync()
            sample = sorted(set([0, C - 1] + rng.integers(0, C, 6).tolist()))
            _checked_chunk(dl, wa, wi, shape, w.seed, T - C, C, sample, layer=li)
            _gather_check(dl, T)
            checked[r] = True
        dl.sync()
        del dl
        torch.cuda.empty_cache()
    assert all(checked.values())
