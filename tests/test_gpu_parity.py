"""GPU parity of every call of the C ABI against the oracle (-m gpu).

Protocol: each call is compared with the oracle run on that call's own inputs
(the GPU state before the call, downloaded): compressed rows and frontier
within rel 2e-3 / abs 1e-4 (the FP8 round trip bit-exact on the GPU's own
pre-quantisation row), indexer scores and top-k bit-exact, attention within
the tolerance, ring commit and checkpoint gather bit-exact.  Sizes span several
tiles with ragged tails; the full-size workloads are checked on sampled outputs.
"""

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs
from gpu_util import (ATOL, RTOL, check_attention_sampled, check_compress, check_indexer_sampled,
                      check_split_mirror, device_layer, download, require_gpu)
from helpers import lane_np, np_in, orc_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    orc.build()


def _run_chunk(dl, wa, wi, shape, seed, pos0, T, report, sample=None, check=True, layer=0):
    """One prefill chunk through all four calls, each checked stage-wise."""
    dev = "cuda"
    h = configs.hidden(shape, seed, T, offset_tok=pos0, layer=layer).to(dev)
    q, q_idx, raw = (x.to(dev) for x in configs.queries(shape, seed, T, offset_tok=pos0, layer=layer))
    before = download(dl) if check else None
    dl.compress_prefill(h, pos0)
    after = download(dl) if check else None
    if check and shape.ratio:
        check_compress(before, after, wa, wi, h.cpu(), pos0, report)
        check_split_mirror(dl)
    topk = None
    n = np.arange(T) if sample is None else np.asarray(sample)
    if shape.ratio == 4:
        V = (pos0 + T) // 4
        topk = torch.empty(T, shape.top_k, dtype=torch.int32, device=dev)
        scores = torch.full((T, max(V, 4)), float("nan"), device=dev)
        dl.indexer_topk(q_idx, [pos0], 1, T, topk, scores, scores.shape[1])
        if check:
            check_indexer_sampled(after, q_idx.cpu().numpy(), [pos0 + j for j in range(T)], topk.cpu().numpy(),
                                  scores.cpu().numpy(), n)
    out = torch.empty(T, shape.n_heads, shape.head_dim, device=dev)
    dl.attention(q, raw, topk, [pos0], 1, T, out, commit_ring=True)
    dl.sync()
    if check:
        check_attention_sampled(after, q.cpu().numpy(), raw.cpu().numpy(),
                                None if topk is None else topk.cpu().numpy(), out.cpu().numpy(), pos0, n)
        # ring commit: slot p % S holds raw row p for the chunk's last min(T, S) positions
        ring = dl.raw[0].cpu().numpy()
        rawc = raw.cpu().numpy()
        for p in range(max(pos0, pos0 + T - shape.swa), pos0 + T):
            np.testing.assert_array_equal(ring[p % shape.swa], rawc[p - pos0])
    return topk, out


def _gather_check(dl, pos):
    n = dl.checkpoint_floats(pos)
    dst = torch.full((n + 8,), float("nan"), device="cuda")
    w = dl.checkpoint_gather(0, pos, dst)
    dl.sync()
    assert w == n
    st = download(dl)
    np.testing.assert_array_equal(dst[:n].cpu().numpy(), orc.checkpoint_gather(st, pos))
    assert torch.isnan(dst[n:]).all()


# ---------------------------------------------------------------------------
# "One ratio-4 layer, 64-token prefill, fp32 throughout, seed 0"
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("splits", [[64], [16, 48], [37, 27]])
def test_c1(splits):
    w = configs.C1
    shape = w.layer
    dl, wa, wi = device_layer(shape, comp_cap=16, idx_cap=16, seed=w.seed)
    report = {}
    pos = 0
    for T in splits:
        _run_chunk(dl, wa, wi, shape, w.seed, pos, T, report)
        pos += T
    _gather_check(dl, pos)
    # the chunk split does not change the state beyond fp32 rounding
    ref, _, _ = device_layer(shape, comp_cap=16, idx_cap=16, seed=w.seed)
    ref.compress_prefill(configs.hidden(shape, w.seed, 64).cuda(), 0)
    torch.cuda.synchronize()
    torch.testing.assert_close(dl.attn_comp, ref.attn_comp, rtol=RTOL, atol=ATOL)
    torch.testing.assert_close(dl.idx_comp, ref.idx_comp, rtol=RTOL, atol=ATOL)


def test_c1_chain_against_oracle_end_to_end():
    """Chain report: the oracle's own end-to-end run (its own state and top-k)."""
    w = configs.C1
    shape = w.layer
    dl, wa, wi = device_layer(shape, comp_cap=16, idx_cap=16, seed=w.seed)
    topk, out = _run_chunk(dl, wa, wi, shape, w.seed, 0, 64, {}, check=False)
    st = orc.State(orc_layer(shape, 16, 16))
    orc.state_init(st)
    orc.compress(st, lane_np(wa), lane_np(wi), np_in(configs.hidden(shape, w.seed, 64)), 0)
    q, q_idx, raw = configs.queries(shape, w.seed, 64)
    tk = orc.indexer_topk(st, q_idx.numpy(), np.arange(64))
    o = orc.attention(st, q.numpy(), raw.numpy(), tk, 0)
    gt = topk.cpu().numpy()
    overlap = np.mean([len(set(a[a >= 0]) & set(b[b >= 0])) / max(1, len(set(b[b >= 0]))) for a, b in zip(gt, tk)])
    assert overlap > 0.95
    same = np.all(gt == tk, axis=1)
    np.testing.assert_allclose(out.cpu().numpy()[same], o[same], rtol=RTOL, atol=ATOL)


# ---------------------------------------------------------------------------
# Multi-tile shapes with ragged tails (D=512, d=128, 64 heads)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ratio,heads,D,swa", [(0, 64, 512, 128), (4, 64, 512, 128), (128, 64, 512, 128),
                                               (4, 32, 512, 128), (4, 64, 128, 128), (4, 64, 256, 128),
                                               (128, 64, 256, 128), (128, 8, 256, 128), (0, 16, 128, 128),
                                               (4, 128, 128, 128), (0, 128, 128, 128), (4, 96, 128, 128),
                                               (4, 64, 512, 64), (0, 64, 256, 32), (128, 32, 512, 100)])
def test_ragged_chunks(ratio, heads, D, swa):
    """heads <= 64: tensor-core attention (head_dim 512, 256 or 128: at 128 the one
    128-wide d-block holds the RoPE dims, so no block is FP8-exact; fewer than 64
    heads run padded to 64 with zero query rows); heads = 128 or 96: groups of 64
    heads.  Rings shorter than 128 rows (swa 64, 32, 100) mask the raw tile's older rows."""
    shape = configs.LayerShape(d_model=512, head_dim=D, n_rot=64, idx_head_dim=128 if D >= 256 else 64,
                               n_heads=heads, ratio=ratio, swa=swa, top_k=16, dtype="bf16", w_std=0.04)
    seed = 21
    T_total = 300 if ratio != 128 else 700
    cap = T_total // max(ratio, 1) + 1
    dl, wa, wi = device_layer(shape, comp_cap=cap, idx_cap=T_total // 4 + 1, seed=seed, gamma_std=0.1)
    report = {}
    pos = 0
    for T in ([131, 169] if ratio != 128 else [131, 300, 269]):
        sample = sorted(set([0, 1, 2, 3, T // 2, T - 2, T - 1] + list(range(0, T, 37))))
        _run_chunk(dl, wa, wi, shape, seed, pos, T, report, sample=sample)
        pos += T
    _gather_check(dl, pos)


# ---------------------------------------------------------------------------
# Decode: B sequences, one token each at staggered positions
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ratio,base,heads,top_k,swa", [(4, 60, 64, 16, 128), (128, 380, 64, 16, 128),
                                                        (0, 200, 64, 16, 128), (4, 60, 8, 16, 128),
                                                        (128, 380, 24, 16, 128), (4, 1600, 64, 384, 128),
                                                        (4, 1600, 24, 1024, 128), (4, 60, 64, 16, 32),
                                                        (0, 28, 64, 16, 32)])
def test_decode_small(ratio, base, heads, top_k, swa):
    """heads < 64: the padded tensor-core attention, split rows combined over the real heads.
    top_k 384: four row tiles, split as the raw tile, two compressed tiles and one.
    top_k 1024: the CUDA-core attention (lists longer than the tensor-core path takes), 24 heads.
    swa 32: a ring shorter than the raw tile (positions 60..67 wrap it; 28..35 fill it)."""
    shape = configs.LayerShape(d_model=512, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=heads, ratio=ratio,
                               swa=swa, top_k=top_k, dtype="bf16", w_std=0.04)
    seed, B = 31, 8
    # every stagger class; ratio 4: some emit this step; ratio 128: 382 + 1 ends a window
    # (383 = 3*128 - 1), the others sit mid-window over 2 visible rows; ratio 0: a wrapped ring
    lens = [base + b for b in range(B)]
    cap = max(lens) // max(ratio, 1) + 2
    icap = max(lens) // 4 + 2
    # the state is built by one prefill per sequence of up to max(lens) tokens
    dl, wa, wi = device_layer(shape, comp_cap=cap, idx_cap=icap, n_seq=B, seed=seed, max_rows=max(lens))
    for b in range(B):
        view = dl.seq_view(b)
        saved = dl.state
        dl.state = view
        h = configs.hidden(shape, seed, lens[b], layer=b).cuda()
        _, _, raw = configs.queries(shape, seed, lens[b], layer=b)
        dl.compress_prefill(h, 0)
        dl.state = saved
        for p in range(max(0, lens[b] - shape.swa), lens[b]):
            dl.raw[b, p % shape.swa] = raw[p].cuda()
    torch.cuda.synchronize()
    befores = [download(dl, b) for b in range(B)]
    hid = torch.stack([configs.hidden(shape, seed, 1, offset_tok=lens[b], layer=b)[0] for b in range(B)]).cuda()
    qs = [configs.queries(shape, seed, 1, offset_tok=lens[b], layer=b) for b in range(B)]
    q = torch.cat([x[0] for x in qs]).cuda()
    q_idx = torch.cat([x[1] for x in qs]).cuda()
    raw = torch.cat([x[2] for x in qs]).cuda()
    dl.compress_decode(hid, lens)
    topk = scores = None
    if ratio == 4:
        topk = torch.empty(B, shape.top_k, dtype=torch.int32, device="cuda")
        vmax = (max(lens) + 1) // 4
        scores = torch.full((B, vmax), float("nan"), device="cuda")
        dl.indexer_topk(q_idx, lens, B, 1, topk, scores, vmax)
    out = torch.empty(B, shape.n_heads, shape.head_dim, device="cuda")
    after_compress = [None] * B
    torch.cuda.synchronize()
    after_compress = [download(dl, b) for b in range(B)]
    dl.attention(q, raw, topk, lens, B, 1, out, commit_ring=True)
    dl.sync()
    for b in range(B):
        if ratio:
            check_compress(befores[b], after_compress[b], wa, wi, hid[b:b + 1].cpu(), lens[b])
        if ratio == 4:
            check_indexer_sampled(after_compress[b], q_idx[b:b + 1].cpu().numpy(), [lens[b]],
                                  topk[b:b + 1].cpu().numpy(), scores[b:b + 1].cpu().numpy(), [0])
        check_attention_sampled(after_compress[b], q[b:b + 1].cpu().numpy(), raw[b:b + 1].cpu().numpy(),
                                None if topk is None else topk[b:b + 1].cpu().numpy(), out[b:b + 1].cpu().numpy(),
                                lens[b], [0])
        np.testing.assert_array_equal(dl.raw[b, lens[b] % shape.swa].cpu().numpy(), raw[b].cpu().numpy())
    if not ratio:
        return
    # decode(t) equals prefill's t-th step: a fresh one-shot prefill of len+1 tokens
    for b in (0, 3):
        ref, _, _ = device_layer(shape, comp_cap=cap, idx_cap=icap, seed=seed)
        ref.compress_prefill(configs.hidden(shape, seed, lens[b] + 1, layer=b).cuda(), 0)
        torch.cuda.synchronize()
        torch.testing.assert_close(dl.attn_comp[b], ref.attn_comp[0], rtol=RTOL, atol=ATOL)
        torch.testing.assert_close(dl.attn_kv[b], ref.attn_kv[0], rtol=RTOL, atol=ATOL)
        if ratio == 4:
            torch.testing.assert_close(dl.idx_comp[b], ref.idx_comp[0], rtol=RTOL, atol=ATOL)


def test_decode_indexer_right_after_prefill_compressor():
    """A decode indexer call straight after prefill compressor calls (no decode compressor in
    between): the score may read rows before waiting for its predecessor only after the decode
    compressor, so here it waits first; scores and lists bit-exact against the oracle."""
    shape = configs.LayerShape(d_model=512, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64, ratio=4,
                               top_k=16, dtype="bf16", w_std=0.04)
    seed, B = 41, 6
    lens = [700 + 37 * b for b in range(B)]                # some (pos + 1) % 4 == 0, some not
    cap = max(lens) // 4 + 2
    dl, wa, wi = device_layer(shape, comp_cap=cap, idx_cap=cap, n_seq=B, seed=seed, max_rows=max(lens))
    for b in range(B):
        view = dl.seq_view(b)
        saved = dl.state
        dl.state = view
        dl.compress_prefill(configs.hidden(shape, seed, lens[b], layer=b).cuda(), 0)
        dl.state = saved
    q_idx = torch.cat([configs.queries(shape, seed, 1, offset_tok=lens[b], layer=b)[1] for b in range(B)]).cuda()
    topk = torch.empty(B, shape.top_k, dtype=torch.int32, device="cuda")
    vmax = (max(lens) + 1) // 4
    scores = torch.full((B, vmax), float("nan"), device="cuda")
    dl.indexer_topk(q_idx, lens, B, 1, topk, scores, vmax)
    dl.sync()
    for b in range(B):
        st = download(dl, b)
        check_indexer_sampled(st, q_idx[b:b + 1].cpu().numpy(), [lens[b]], topk[b:b + 1].cpu().numpy(),
                              scores[b:b + 1].cpu().numpy(), [0])


# ---------------------------------------------------------------------------
# "One ratio-128 layer, 8192-token prefill in two 4096-token chunks" (full size)
# ---------------------------------------------------------------------------

def test_c2_full():
    w = configs.C2
    shape = w.layer
    dl, wa, wi = device_layer(shape, comp_cap=w.n_tok // 128, seed=w.seed)
    report = {}
    for c in range(w.n_tok // w.chunk):
        sample = [0, 1, 127, 128, 1000, 2047, 4094, 4095]
        _run_chunk(dl, wa, wi, shape, w.seed, c * w.chunk, w.chunk, report, sample=sample)
    _gather_check(dl, w.n_tok)


def test_decode_one_sequence_short_prefix():
    """A one-sequence layer whose workspace was sized for 4-token prefill chunks
    takes a decode step: the workspace size covers decode steps of the layer's
    sequence count (the decode layout's split partials exceed such a prefill's)."""
    shape = configs.LayerShape(d_model=520, head_dim=128, n_rot=32, idx_head_dim=128, n_heads=16, ratio=4,
                               top_k=512, dtype="f32", w_std=0.04)
    seed = 61
    dl, wa, wi = device_layer(shape, comp_cap=8, idx_cap=8, n_seq=1, seed=seed, max_rows=4)
    h = configs.hidden(shape, seed, 7).cuda()
    q, q_idx, raw = (x.cuda() for x in configs.queries(shape, seed, 7))
    dl.compress_prefill(h[:3], 0)
    dl.compress_prefill(h[3:6], 3)
    dl.raw[0, :6] = raw[:6]
    torch.cuda.synchronize()
    before = download(dl)
    dl.compress_decode(h[6:7], [6])
    topk = torch.empty(1, shape.top_k, dtype=torch.int32, device="cuda")
    scores = torch.full((1, 4), float("nan"), device="cuda")
    dl.indexer_topk(q_idx[6:7], [6], 1, 1, topk, scores, 4)
    out = torch.empty(1, shape.n_heads, shape.head_dim, device="cuda")
    torch.cuda.synchronize()
    after = download(dl)
    dl.attention(q[6:7], raw[6:7], topk, [6], 1, 1, out, commit_ring=True)
    dl.sync()
    check_compress(before, after, wa, wi, h[6:7].cpu(), 6)
    check_indexer_sampled(after, q_idx[6:7].cpu().numpy(), [6], topk.cpu().numpy(), scores.cpu().numpy(), [0])
    check_attention_sampled(after, q[6:7].cpu().numpy(), raw[6:7].cpu().numpy(), topk.cpu().numpy(),
                            out.cpu().numpy(), 6, [0])


# ---------------------------------------------------------------------------
# Checkpoint restore: gather -> scatter into a fresh state -> continue
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ratio,heads,D", [(4, 64, 512), (128, 64, 512), (0, 64, 512), (4, 8, 128)])
def test_checkpoint_restore_resumes_bit_exact(ratio, heads, D):
    """Restored state equals the saved one on every live region (and the bf16
    mirror is rebuilt), and continuing from it gives the uninterrupted run's
    outputs bit for bit; the oracle's restore of the same body agrees."""
    dtype = "bf16" if D == 512 else "f32"
    shape = configs.LayerShape(d_model=512 if D == 512 else 256, head_dim=D, n_rot=64, idx_head_dim=128 if D == 512 else 64,
                               n_heads=heads, ratio=ratio, top_k=16, dtype=dtype, w_std=0.04)
    seed, T1, T2 = 41, 301, 170                       # T1 is mid-window for both ratios and wraps the ring
    cap = (T1 + T2) // max(ratio, 1) + 1
    icap = (T1 + T2) // 4 + 1
    dl, wa, wi = device_layer(shape, comp_cap=cap, idx_cap=icap, seed=seed)
    _run_chunk(dl, wa, wi, shape, seed, 0, T1, {}, check=False)
    n = dl.checkpoint_floats(T1)
    body = torch.empty(n, device="cuda")
    dl.checkpoint_gather(0, T1, body)
    dl.sync()
    # restore into a fresh layer (same weights)
    fresh, _, _ = device_layer(shape, comp_cap=cap, idx_cap=icap, seed=seed)
    fresh.checkpoint_scatter(0, T1, body)
    fresh.sync()
    again = torch.empty(n, device="cuda")
    fresh.checkpoint_gather(0, T1, again)
    fresh.sync()
    assert torch.equal(again, body)
    if ratio and dl.attn_split is not None:
        rows = T1 // ratio
        assert torch.equal(fresh.attn_split[:, :rows], dl.attn_split[:, :rows])
    # the oracle restores the same body to the same gather
    st = orc.State(orc_layer(shape, cap, icap))
    orc.state_init(st)
    orc.checkpoint_scatter(st, T1, body.cpu().numpy())
    np.testing.assert_array_equal(orc.checkpoint_gather(st, T1), body.cpu().numpy())
    # continue both with the same chunk
    tk_a, out_a = _run_chunk(dl, wa, wi, shape, seed, T1, T2, {}, check=False)
    tk_b, out_b = _run_chunk(fresh, wa, wi, shape, seed, T1, T2, {}, check=False)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    if tk_a is not None:
        assert torch.equal(tk_a, tk_b)
    n2 = dl.checkpoint_floats(T1 + T2)
    ga, gb = torch.empty(n2, device="cuda"), torch.empty(n2, device="cuda")
    dl.checkpoint_gather(0, T1 + T2, ga)
    fresh.checkpoint_gather(0, T1 + T2, gb)
    dl.sync()
    assert torch.equal(ga, gb)


# ---------------------------------------------------------------------------
# Top-k on crafted index rows: heavy ties (the radix path), a few distinct
# scores (ties inside the boundary bin), signed zeros, a few strided stretches
# of high rows, V around k and across the bitmap word boundaries; scores and
# lists bit-exact against the oracle
# ---------------------------------------------------------------------------

_TK_SHAPE = configs.LayerShape(d_model=256, head_dim=128, n_rot=64, idx_head_dim=64, n_heads=8, ratio=4, top_k=512,
                               dtype="f32")
_TK_CAP = 8200


def _crafted_rows(kind, n, d, rng):
    if kind in ("random", "zero_query"):
        return rng.standard_normal((n, d)).astype(np.float32)
    if kind == "all_equal":
        return np.tile(rng.integers(-3, 4, d).astype(np.float32), (n, 1))
    if kind == "few_values":
        base = rng.integers(-3, 4, (5, d)).astype(np.float32)
        return base[rng.integers(0, 5, n)]
    if kind == "signed_zero":
        r = np.zeros((n, d), np.float32)
        r[:, 0] = rng.choice(np.array([-0.0, 0.0, 1.0, -1.0, 2.0], np.float32), n)
        return r
    if kind == "skewed":
        # high rows in eight short stretches, fewer than k of them in all
        r = rng.standard_normal((n, d)).astype(np.float32)
        for st in range(8):
            r[st * 1024 + 8:st * 1024 + 120] += 4.0
            r[st * 512 + 4:st * 512 + 28] += 4.0
        return r
    raise ValueError(kind)


def _crafted_queries(kind, n, d, rng):
    if kind == "zero_query":
        return np.zeros((n, d), np.float32)
    if kind == "random":
        return rng.standard_normal((n, d)).astype(np.float32)
    if kind == "skewed":
        return rng.integers(0, 3, (n, d)).astype(np.float32)  # non-negative: the raised rows score high
    return rng.integers(-2, 3, (n, d)).astype(np.float32)    # integer scores: ties stay exact


_TK_KINDS = ["random", "all_equal", "few_values", "signed_zero", "zero_query", "skewed"]


@pytest.mark.parametrize("kind", _TK_KINDS)
def test_topk_crafted_rows_prefill(kind):
    shape = _TK_SHAPE
    d, k = shape.idx_head_dim, shape.top_k
    rng = np.random.default_rng(_TK_KINDS.index(kind) + 70)
    dl, _, _ = device_layer(shape, comp_cap=16, idx_cap=_TK_CAP, seed=5, max_rows=64)
    dl.idx_comp[0] = torch.from_numpy(_crafted_rows(kind, _TK_CAP, d, rng)).cuda()
    st = download(dl)
    # V = (pos + 1) / 4 runs over k - 1 .. k + 4, 4094 .. 4098 and 8189 .. 8193
    for pos0, T in ((4 * k - 5, 24), (4 * 4096 - 6, 16), (4 * 8190 - 3, 12)):
        q_idx = _crafted_queries(kind, T, d, rng)
        V = (pos0 + T) // 4
        topk = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        scores = torch.full((T, V), float("nan"), device="cuda")
        dl.indexer_topk(torch.from_numpy(q_idx).cuda(), [pos0], 1, T, topk, scores, V)
        dl.sync()
        check_indexer_sampled(st, q_idx, [pos0 + j for j in range(T)], topk.cpu().numpy(), scores.cpu().numpy(),
                              range(T))


@pytest.mark.parametrize("kind", ["random", "all_equal", "few_values"])
def test_topk_crafted_rows_decode(kind):
    shape = _TK_SHAPE
    d, k = shape.idx_head_dim, shape.top_k
    rng = np.random.default_rng(["random", "all_equal", "few_values"].index(kind) + 90)
    lens = [4 * k - 5, 4 * k + 3, 4095, 16383, 16390, 32770]       # V = 511, 513, 1024, 4096, 4097, 8192
    B = len(lens)
    dl, _, _ = device_layer(shape, comp_cap=16, idx_cap=_TK_CAP, n_seq=B, seed=5, max_rows=64)
    for b in range(B):
        dl.idx_comp[b] = torch.from_numpy(_crafted_rows(kind, _TK_CAP, d, rng)).cuda()
    q_idx = _crafted_queries(kind, B, d, rng)
    vmax = max((p + 1) // 4 for p in lens)
    topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, vmax), float("nan"), device="cuda")
    dl.indexer_topk(torch.from_numpy(q_idx).cuda(), lens, B, 1, topk, scores, vmax)
    dl.sync()
    for b in range(B):
        check_indexer_sampled(download(dl, b), q_idx[b:b + 1], [lens[b]], topk[b:b + 1].cpu().numpy(),
                              scores[b:b + 1].cpu().numpy(), [0])


@pytest.mark.parametrize("kind", ["random", "few_values"])
def test_topk_decode_long_rows(kind):
    """Decode top-k over 28.9K-40960 visible rows, where the keys no longer fit
    shared memory and each pass reads the score row again (few_values also
    overflows the candidate list, so the radix path runs on 1024 threads)."""
    shape = _TK_SHAPE
    d, k = shape.idx_head_dim, shape.top_k
    cap = 40960
    rng = np.random.default_rng(["random", "few_values"].index(kind) + 110)
    lens = [4 * 28900 - 1, 4 * 30001 + 1, 4 * cap - 1]              # V = 28900, 30001, 40960
    B = len(lens)
    dl, _, _ = device_layer(shape, comp_cap=16, idx_cap=cap, n_seq=B, seed=5, max_rows=64)
    for b in range(B):
        dl.idx_comp[b] = torch.from_numpy(_crafted_rows(kind, cap, d, rng)).cuda()
    q_idx = _crafted_queries(kind, B, d, rng)
    vmax = max((p + 1) // 4 for p in lens)
    topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, vmax), float("nan"), device="cuda")
    dl.indexer_topk(torch.from_numpy(q_idx).cuda(), lens, B, 1, topk, scores, vmax)
    dl.sync()
    for b in range(B):
        check_indexer_sampled(download(dl, b), q_idx[b:b + 1], [lens[b]], topk[b:b + 1].cpu().numpy(),
                              scores[b:b + 1].cpu().numpy(), [0])


def _chain_layer(n_seq, d):
    """Rows and queries built from vectors on which the in-order fused chain differs
    from the reversed chain, the unfused chain and a dot rounded once; each vector is
    zero-padded after its last dimension (which leaves every chain's value as it is)."""
    from fp_exact import distinguishing_pairs
    pairs = [p for w in (4, 6, 8) for p in distinguishing_pairs(6, w, seed=300 + w)]
    rows = np.zeros((len(pairs), d), np.float32)
    qs = np.zeros((len(pairs), d), np.float32)
    for i, (q, r, _) in enumerate(pairs):
        rows[i, :len(r)] = r
        qs[i, :len(q)] = q
    return pairs, rows, qs


def test_index_score_chain_vectors_prefill_and_decode():
    """The GPU scores are the in-order binary32 fmaf chain, computed here in exact
    arithmetic, on vectors where the other plausible evaluation orders differ."""
    from fp_exact import fma_chain
    shape = _TK_SHAPE
    d = shape.idx_head_dim
    pairs, rows, qs = _chain_layer(1, d)
    n = len(pairs)
    cap = 80
    rng = np.random.default_rng(400)
    full = np.concatenate([rows, rng.standard_normal((cap - n, d)).astype(np.float32)])
    want = np.array([[fma_chain(qs[j], full[c]) for c in range(cap)] for j in range(n)], np.float32)
    for j in range(n):
        assert want[j, j] == pairs[j][2]
    # prefill form: n queries of one sequence at positions 255 .. 255 + n - 1 (64 .. 68 visible rows)
    dl, _, _ = device_layer(shape, comp_cap=16, idx_cap=cap, seed=5, max_rows=64)
    dl.idx_comp[0] = torch.from_numpy(full).cuda()
    pos0 = 255
    topk = torch.full((n, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((n, cap), float("nan"), device="cuda")
    dl.indexer_topk(torch.from_numpy(qs).cuda(), [pos0], 1, n, topk, scores, cap)
    dl.sync()
    sc = scores.cpu().numpy()
    for j in range(n):
        V = (pos0 + j + 1) // 4
        np.testing.assert_array_equal(sc[j, :V], want[j, :V], err_msg=f"prefill scores query {j}")
    st = download(dl)
    check_indexer_sampled(st, qs, [pos0 + j for j in range(n)], topk.cpu().numpy(), sc, range(n))
    # decode form: one query per sequence (TMA-staged score), every sequence holding the same rows
    B = n
    dd, _, _ = device_layer(shape, comp_cap=16, idx_cap=cap, n_seq=B, seed=5, max_rows=64)
    for b in range(B):
        dd.idx_comp[b] = torch.from_numpy(full).cuda()
    lens = [4 * cap - 1 - (b % 3) for b in range(B)]
    topk = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, cap), float("nan"), device="cuda")
    dd.indexer_topk(torch.from_numpy(qs).cuda(), lens, B, 1, topk, scores, cap)
    dd.sync()
    sc = scores.cpu().numpy()
    for b in range(B):
        V = (lens[b] + 1) // 4
        np.testing.assert_array_equal(sc[b, :V], want[b, :V], err_msg=f"decode scores sequence {b}")
        check_indexer_sampled(download(dd, b), qs[b:b + 1], [lens[b]], topk[b:b + 1].cpu().numpy(), sc[b:b + 1],
                              [0])
