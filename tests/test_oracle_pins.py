"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test ties one oracle function to something other than itself: a value the
pages print (golden fixtures), a closed form, an invariant the spec lists,
a library routine (numpy matmul, torch's float8_e4m3fn cast) or brute force.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from compressed_kv_sparse_compressor_gb300 import configs, synth
from helpers import (dense_attention, e4m3_torch, fp8_rows_window_form, lane_np, np_in,
                     orc_layer, window_form_lane)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Routing, ring capacity, chunk size (values printed on the pages)
# --------------------------------------------------------------------------

def test_layer_ratio_tables(orc):
    g = _golden("layer_ratios.json")
    assert [orc.layer_ratio(0, i) for i in range(10)] == g["flash"]
    assert [orc.layer_ratio(1, i) for i in range(10)] == g["pro"]
    assert tuple(g["flash"][:8]) == configs.C3.ratios


def test_raw_cap_and_chunk(orc):
    g = _golden("schedule_constants.json")
    for ctx, cap in g["raw_cap"]:
        assert orc.raw_cap(ctx) == cap
    for n, c in g["prefill_chunk_no_env"]:
        assert orc.prefill_chunk(n) == c
    for n, env, c in g["prefill_chunk_env"]:
        assert orc.prefill_chunk(n, env) == c
    assert g["head_dim"] - g["n_rot"] == g["n_nope"]
    s = configs.C5.layer
    assert (s.head_dim, s.n_rot, s.idx_head_dim, s.top_k, s.swa) == (
        g["head_dim"], g["n_rot"], g["idx_head_dim"], g["top_k"], 128)


def test_inv_freq_closed_form(orc):
    for R in (64, 16):
        f = orc.inv_freq(10000.0, R)
        assert f[0] == 1.0
        i = np.arange(R // 2)
        expect = np.exp(-2.0 * i / R * math.log(10000.0))
        np.testing.assert_allclose(f, expect, rtol=2 ** -23)
        assert np.all(np.diff(f) < 0)


# --------------------------------------------------------------------------
# A1 projections
# --------------------------------------------------------------------------

@pytest.mark.parametrize("bf16", [False, True])
def test_project_matches_matmul(orc, bf16):
    dt = torch.bfloat16 if bf16 else torch.float32
    W = synth.normal(1, 100, (48, 96), std=0.05, dtype=dt)
    h = synth.normal(1, 101, (7, 96), dtype=dt)
    out = orc.project(np_in(W), np_in(h), bf16=bf16)
    ref = (h.double() @ W.double().T).float().numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------
# A7 FP8 E4M3 round trip
# --------------------------------------------------------------------------

def test_e4m3_format_golden(orc):
    g = _golden("e4m3fn_format.json")
    for y, want in g["round_cases"]:
        assert orc.e4m3_rne(np.float32(y)) == np.float32(want), y
    assert orc.e4m3_rne(np.float32(g["max_normal"])) == g["max_normal"]
    assert orc.e4m3_rne(np.float32(g["min_subnormal"])) == g["min_subnormal"]
    for v in g["values_1_to_2"]:
        assert orc.e4m3_rne(np.float32(v)) == v


def test_e4m3_matches_torch_cast(orc):
    rng = np.random.default_rng(7)
    grid = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    mids = (grid[:-1].astype(np.float64) + grid[1:]) / 2
    ys = np.concatenate([
        grid, -grid, mids.astype(np.float32), -mids.astype(np.float32),
        (rng.standard_normal(4000) * 10.0 ** rng.uniform(-3, 2.6, 4000)).astype(np.float32),
    ])
    ys = np.clip(ys, -448, 448).astype(np.float32)
    got = orc.e4m3_rne(ys)
    np.testing.assert_array_equal(got, e4m3_torch(ys))


def test_fp8_scale_exponent(orc):
    rng = np.random.default_rng(3)
    for a in np.concatenate([10.0 ** rng.uniform(-6, 6, 500), [448.0, 224.0, 1.0, 896.0, 448.000031]]):
        a = np.float32(a)
        e = orc.fp8_scale_exp(a)
        assert a <= 448.0 * 2.0 ** e and a > 448.0 * 2.0 ** (e - 1)
    assert orc.fp8_scale_exp(0.0) == 0


def test_fp8_roundtrip_properties(orc):
    rng = np.random.default_rng(11)
    rows = (rng.standard_normal((6, 512)) * rng.uniform(0.01, 50, (6, 1))).astype(np.float32)
    rows[3, 64:128] = 0.0
    out = orc.fp8_roundtrip(rows, 448)
    np.testing.assert_array_equal(out[:, 448:], rows[:, 448:])          # RoPE tail untouched
    np.testing.assert_array_equal(out[3, 64:128], 0.0)
    for i in range(6):
        for b in range(7):
            blk, src = out[i, 64 * b:64 * b + 64], rows[i, 64 * b:64 * b + 64]
            e = orc.fp8_scale_exp(np.max(np.abs(src)))
            y = blk.astype(np.float64) * 2.0 ** -e
            np.testing.assert_array_equal(e4m3_torch(y.astype(np.float32)), y)   # on the grid
            assert np.all(np.abs(blk - src) <= np.abs(src) * 2 ** -4 + 2.0 ** (e - 10))
    np.testing.assert_array_equal(orc.fp8_roundtrip(out, 448), out)        # fixed points
    np.testing.assert_array_equal(out, fp8_rows_window_form(rows, 448))


# --------------------------------------------------------------------------
# A5 RMSNorm, A6 tail RoPE
# --------------------------------------------------------------------------

def test_rmsnorm_closed_form(orc):
    for c in (3.0, -0.5, 1e-4):
        x = np.full(64, c)
        y = orc.rmsnorm(x, eps=1e-6)
        eps = float(np.float32(1e-6))           # the config carries eps as a float
        np.testing.assert_allclose(y, c / math.sqrt(c * c + eps), rtol=1e-13)
    g = np.linspace(0.5, 1.5, 64).astype(np.float32)
    y = orc.rmsnorm(np.full(64, 2.0), g, eps=0.0)
    np.testing.assert_allclose(y, g.astype(np.float64), rtol=1e-13)


def test_rope_tail_properties(orc):
    R, D = 64, 512
    f = orc.inv_freq(10000.0, R)
    rng = np.random.default_rng(5)
    x = rng.standard_normal(D)
    for p in (0, 1, 4, 131068):
        y = orc.rope_tail(x, R, p, f)
        np.testing.assert_array_equal(y[:D - R], x[:D - R])
        np.testing.assert_allclose(np.linalg.norm(y[D - R:]), np.linalg.norm(x[D - R:]), rtol=1e-12)
        pairs_in = x[D - R:].reshape(-1, 2)
        pairs_out = y[D - R:].reshape(-1, 2)
        np.testing.assert_allclose(np.linalg.norm(pairs_out, axis=1), np.linalg.norm(pairs_in, axis=1), rtol=1e-12)
    np.testing.assert_array_equal(orc.rope_tail(x, R, 0, f), x)
    # one nonzero tail dim 2i rotates into (2i, 2i+1) by the angle float32(p * theta_i)
    for i in (0, 5, 31):
        e = np.zeros(D)
        e[D - R + 2 * i] = 1.0
        p = 1000
        y = orc.rope_tail(e, R, p, f)
        ang = float(np.float32(np.float32(p) * f[i]))
        want = np.zeros(D)
        want[D - R + 2 * i] = math.cos(ang)
        want[D - R + 2 * i + 1] = math.sin(ang)
        np.testing.assert_allclose(y, want, atol=1e-15)
    # relative-position property: <rope(a, p), rope(b, p + 8)> does not depend on p
    a, b = rng.standard_normal(D), rng.standard_normal(D)
    dots = [np.dot(orc.rope_tail(a, R, p, f)[D - R:], orc.rope_tail(b, R, p + 8, f)[D - R:])
            for p in (0, 8, 64)]
    np.testing.assert_allclose(dots, dots[0], rtol=1e-5)


# --------------------------------------------------------------------------
# A2-A8 compressor
# --------------------------------------------------------------------------

def _small_shape(ratio, dtype="f32", D=128, d=64, R=64, dm=96):
    return configs.LayerShape(d_model=dm, head_dim=D, n_rot=R, idx_head_dim=d, n_heads=4, ratio=ratio,
                              top_k=8, dtype=dtype, w_std=1.0 / 16)


def test_pool_equal_scores_is_mean(orc):
    """spec invariant 1: equal scores make the pool the mean of its candidates."""
    shape = _small_shape(4)
    L = orc_layer(shape, comp_cap=8)
    st = orc.State(L)
    orc.state_init(st)
    D = shape.head_dim
    rng = np.random.default_rng(1)
    ape = np.full((4, 2 * D), 0.25, np.float32)
    kvs = rng.standard_normal((12, 2 * D)).astype(np.float32)
    f = orc.inv_freq(shape.rope_base, shape.n_rot)
    for p in range(12):
        orc.compress_token(L, True, ape, None, st.attn, kvs[p], np.zeros(2 * D, np.float32), p)
    # window 0: rows 0..3 are the fresh frontier (score -inf), so 4 candidates
    means = [kvs[0:4, D:].mean(0)]
    for c in (1, 2):
        means.append(np.concatenate([kvs[4 * (c - 1):4 * c, :D], kvs[4 * c:4 * c + 4, D:]]).mean(0))
    for c, m in enumerate(means):
        want = orc.rope_tail(orc.rmsnorm(m.astype(np.float64), None, shape.rms_eps), shape.n_rot, 4 * c, f)
        np.testing.assert_allclose(st.attn.prequant[c], want.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_pool_two_candidates_closed_form(orc):
    shape = _small_shape(128, D=64, R=16)
    L = orc_layer(shape, comp_cap=2)
    st = orc.State(L)
    orc.state_init(st)
    D = shape.head_dim
    kv = np.zeros((128, D), np.float32)
    sc = np.full((128, D), -1e30, np.float32)
    kv[5], kv[77] = 1.0, -2.0
    sc[5], sc[77] = 0.3, 1.1
    ape = np.zeros((128, D), np.float32)
    for p in range(128):
        orc.compress_token(L, True, ape, None, st.attn, kv[p], sc[p], p)
    w5, w77 = math.exp(0.3 - 1.1), 1.0
    pooled = (w5 * 1.0 + w77 * -2.0) / (w5 + w77)
    # constant row -> RMSNorm gives sign(pooled) * |pooled| / sqrt(pooled^2 + eps); p = 0 -> no rotation
    want = pooled / math.sqrt(pooled * pooled + float(np.float32(shape.rms_eps)))
    np.testing.assert_allclose(st.attn.prequant[0], want, rtol=1e-6)


def test_shift_and_first_window(orc):
    shape = _small_shape(4)
    L = orc_layer(shape, comp_cap=4)
    st = orc.State(L)
    orc.state_init(st)
    D = shape.head_dim
    rng = np.random.default_rng(2)
    ape = rng.standard_normal((4, 2 * D)).astype(np.float32)
    kvs = rng.standard_normal((8, 2 * D)).astype(np.float32)
    scs = rng.standard_normal((8, 2 * D)).astype(np.float32)
    for p in range(3):
        orc.compress_token(L, True, ape, None, st.attn, kvs[p], scs[p], p)
    assert np.all(np.isneginf(st.attn.state_score[:4])) and np.all(st.attn.state_kv[:4] == 0)
    orc.compress_token(L, True, ape, None, st.attn, kvs[3], scs[3], 3)
    # after the boundary rows 0..3 are a copy of rows 4..7 (tokens 0..3)
    np.testing.assert_array_equal(st.attn.state_kv[:4], st.attn.state_kv[4:])
    np.testing.assert_array_equal(st.attn.state_kv[:4], kvs[:4])
    np.testing.assert_array_equal(st.attn.state_score[:4], (scs[:4] + ape).astype(np.float32))
    # first window pools the current half only: softmax over rows 4..7 at columns D..2D
    s = (scs[:4, D:] + ape[:, D:]).astype(np.float64)
    w = np.exp(s - s.max(0))
    pooled = (w * kvs[:4, D:]).sum(0) / w.sum(0)
    f = orc.inv_freq(shape.rope_base, shape.n_rot)
    want = orc.rope_tail(orc.rmsnorm(pooled, None, shape.rms_eps), shape.n_rot, 0, f)
    np.testing.assert_allclose(st.attn.prequant[0], want.astype(np.float32), rtol=1e-6, atol=1e-7)


def _run_compress(orc, shape, w_attn, w_idx, hidden, splits, comp_cap, idx_cap):
    L = orc_layer(shape, comp_cap, idx_cap)
    st = orc.State(L)
    orc.state_init(st)
    p = 0
    for n in splits:
        orc.compress(st, lane_np(w_attn), lane_np(w_idx) if w_idx else None, np_in(hidden[p:p + n]), p)
        p += n
    return st


@pytest.mark.parametrize("ratio,T", [(4, 64), (4, 67), (128, 300)])
def test_row_count_and_chunk_invariance(orc, ratio, T):
    """spec invariants 2 and 3: T // ratio rows; any chunk split gives identical results."""
    shape = _small_shape(ratio)
    seed = 0
    w_attn = configs.lane_weights(shape, seed, 0, "attn", gamma_std=0.1)
    w_idx = configs.lane_weights(shape, seed, 0, "idx", gamma_std=0.1) if ratio == 4 else None
    h = configs.hidden(shape, seed, T)
    cap = T // ratio + 2
    icap = T // 4 + 2 if ratio == 4 else 0
    ref = _run_compress(orc, shape, w_attn, w_idx, h, [T], cap, icap)
    n_rows = T // ratio
    assert not np.isnan(ref.attn.comp[:n_rows]).any() and np.isnan(ref.attn.comp[n_rows:]).all()
    if ratio == 4:
        assert not np.isnan(ref.idx.comp[:T // 4]).any() and np.isnan(ref.idx.comp[T // 4:]).all()
    splits_list = [[16, T - 16], [37, T - 37], [1] * 9 + [T - 9]]
    for splits in splits_list:
        st = _run_compress(orc, shape, w_attn, w_idx, h, splits, cap, icap)
        for a, b in ((st.attn, ref.attn), (st.idx, ref.idx)):
            np.testing.assert_array_equal(a.comp, b.comp)
            np.testing.assert_array_equal(a.prequant, b.prequant)
            np.testing.assert_array_equal(a.state_kv, b.state_kv)
            np.testing.assert_array_equal(a.state_score, b.state_score)


@pytest.mark.parametrize("ratio,T,dtype", [(4, 64, "f32"), (4, 66, "bf16"), (128, 300, "f32")])
def test_compressor_matches_window_form(orc, ratio, T, dtype):
    """Brute force: rows formed directly from each window's tokens equal the frontier recurrence."""
    shape = _small_shape(ratio, dtype=dtype)
    seed = 9
    w_attn = configs.lane_weights(shape, seed, 0, "attn", gamma_std=0.1)
    w_idx = configs.lane_weights(shape, seed, 0, "idx", gamma_std=0.1) if ratio == 4 else None
    h = configs.hidden(shape, seed, T)
    st = _run_compress(orc, shape, w_attn, w_idx, h, [T], T // ratio, T // 4 if ratio == 4 else 0)
    n = T // ratio
    pre, fin, kv, sa = window_form_lane(shape, w_attn, h, True)
    np.testing.assert_allclose(st.attn.prequant[:n], pre, rtol=1e-5, atol=1e-6)
    # FP8 of the oracle's own pre-quant rows, done independently, is bit-identical
    np.testing.assert_array_equal(st.attn.comp[:n], fp8_rows_window_form(st.attn.prequant[:n], shape.head_dim - shape.n_rot))
    # frontier after T tokens, from the window form
    m = T % ratio
    if ratio == 4:
        base = T - m
        for q in range(4):
            np.testing.assert_allclose(st.attn.state_kv[q], kv[base - 4 + q], rtol=1e-6, atol=1e-6)
            np.testing.assert_allclose(st.attn.state_score[q], sa[base - 4 + q], rtol=1e-6, atol=1e-6)
            src = base + q if q < m else base - 4 + q
            np.testing.assert_allclose(st.attn.state_kv[4 + q], kv[src], rtol=1e-6, atol=1e-6)
        ipre, ifin, _, _ = window_form_lane(shape, w_idx, h, False)
        np.testing.assert_allclose(st.idx.comp[:T // 4], ipre, rtol=1e-5, atol=1e-6)
        np.testing.assert_array_equal(st.idx.comp[:T // 4], st.idx.prequant[:T // 4])
    else:
        for q in range(ratio):
            src = (T - m) + q if q < m else (T - m) - ratio + q
            np.testing.assert_allclose(st.attn.state_kv[q], kv[src], rtol=1e-6, atol=1e-6)
            np.testing.assert_allclose(st.attn.state_score[q], sa[src], rtol=1e-6, atol=1e-6)


# --------------------------------------------------------------------------
# A9-A10 indexer score and top-k
# --------------------------------------------------------------------------

def test_index_score_error_bound(orc):
    rng = np.random.default_rng(4)
    for d in (64, 128):
        for _ in range(200):
            q = rng.standard_normal(d).astype(np.float32)
            r = rng.standard_normal(d).astype(np.float32)
            s = orc.index_score(q, r)
            exact = float(np.dot(q.astype(np.float64), r.astype(np.float64)))
            bound = d * 2.0 ** -24 * float(np.sum(np.abs(q.astype(np.float64) * r)))
            assert abs(s - exact) <= bound
            assert np.float32(s) == s


def test_round_f32_rule():
    """The exact-rounding helper itself: ties to even, subnormal quantum, exact values kept."""
    from fractions import Fraction as Fr

    from fp_exact import round_f32
    u = Fr(1, 1 << 24)                                   # half an ulp of 1.0
    assert round_f32(1 + u) == np.float32(1.0)            # tie -> even significand
    assert round_f32(1 + 3 * u) == np.float32(1.0) + np.float32(2.0 ** -22)
    assert round_f32(1 + u + Fr(1, 1 << 60)) == np.float32(1.0) + np.float32(2.0 ** -23)
    assert round_f32(-(1 + 3 * u)) == -(np.float32(1.0) + np.float32(2.0 ** -22))
    assert round_f32(Fr(1, 1 << 150)) == 0.0             # half the smallest subnormal -> 0 (even)
    assert round_f32(Fr(3, 1 << 150)) == np.float32(2.0 ** -148)
    rng = np.random.default_rng(12)
    for x in rng.standard_normal(500).astype(np.float32):
        assert round_f32(Fr(float(x))) == x
    for x in rng.standard_normal(500):                     # doubles: numpy's cast rounds to nearest even too
        assert round_f32(Fr(float(x))) == np.float32(x)


def test_index_score_is_the_in_order_fused_chain(orc):
    """The indexer score is s = fmaf(q[i], row[i], s) for i = 0..d-1 in binary32
    (the reading that makes the top-k bit-exact).  On crafted vectors the in-order
    fused chain, the reversed chain, the unfused chain, the exact dot rounded once
    and a double accumulation give different binary32 results; the oracle must give
    the first, computed here in exact rational arithmetic."""
    from fp_exact import distinguishing_pairs
    for d in (4, 6, 8):
        for q, r, want in distinguishing_pairs(6, d, seed=300 + d):
            got = np.float32(orc.index_score(q, r))
            assert got == want, (d, q.tolist(), r.tolist(), float(got), float(want))
            # zero padding after the last dimension leaves the chain's value unchanged
            qp = np.concatenate([q, np.zeros(128 - d, np.float32)])
            rp = np.concatenate([r, rng_pad(128 - d)])
            assert np.float32(orc.index_score(qp, rp)) == want


def rng_pad(n):
    return np.random.default_rng(n).standard_normal(n).astype(np.float32)


def test_topk_brute_force(orc):
    rng = np.random.default_rng(6)
    for trial in range(300):
        V = int(rng.integers(0, 40))
        k = int(rng.integers(1, 12))
        vals = np.array([-1.5, -0.0, 0.0, 0.5, 2.0, 3.25], np.float32)
        s = rng.choice(vals, size=max(V, 1)).astype(np.float32)
        got = orc.topk(s, V, k)
        order = sorted(range(V), key=lambda c: (-float(s[c]), c))[:k]
        want = sorted(order) + [-1] * (k - min(k, V))
        assert got.tolist() == want


def test_indexer_topk_visibility(orc):
    shape = _small_shape(4)
    L = orc_layer(shape, comp_cap=16, idx_cap=16)
    st = orc.State(L)
    rng = np.random.default_rng(8)
    st.idx.comp[:] = rng.standard_normal(st.idx.comp.shape).astype(np.float32)
    pos = np.arange(0, 64)
    q = rng.standard_normal((64, shape.idx_head_dim)).astype(np.float32)
    tk, sc = orc.indexer_topk(st, q, pos, want_scores=True)
    for j, t in enumerate(pos):
        V = (t + 1) // 4
        s = [orc.index_score(q[j], st.idx.comp[c]) for c in range(V)]
        want = sorted(sorted(range(V), key=lambda c: (-s[c], c))[:shape.top_k])
        assert tk[j].tolist() == want + [-1] * (shape.top_k - len(want))
        np.testing.assert_array_equal(sc[j, :V], np.array(s, np.float32))


# --------------------------------------------------------------------------
# A11 attention, A12 ring commit
# --------------------------------------------------------------------------

def _attn_state(orc, ratio, T_prev=0, S=16, D=64, H=3, k=6, cap=40):
    shape = configs.LayerShape(d_model=32, head_dim=D, n_rot=16, idx_head_dim=16, n_heads=H, ratio=ratio,
                               swa=S, top_k=k, dtype="f32")
    L = orc_layer(shape, comp_cap=cap, idx_cap=cap)
    st = orc.State(L)
    rng = np.random.default_rng(ratio + 100)
    st.attn.comp[:] = rng.standard_normal(st.attn.comp.shape).astype(np.float32)
    st.raw[:] = rng.standard_normal(st.raw.shape).astype(np.float32)
    return shape, L, st, rng


@pytest.mark.parametrize("ratio", [0, 4, 128])
def test_attention_k_all_is_dense(orc, ratio):
    """spec invariant 6: with every visible row selected the result is dense attention."""
    S = 16
    shape, L, st, rng = _attn_state(orc, ratio, S=S, k=64, cap=64)
    pos0, T = 200, 60
    if ratio == 128:
        pos0, T = 250, 20           # crosses the emit at position 255
    q = rng.standard_normal((T, shape.n_heads, shape.head_dim)).astype(np.float32)
    raw_new = rng.standard_normal((T, shape.head_dim)).astype(np.float32)
    tk = None
    if ratio == 4:
        tk = np.full((T, 64), -1, np.int32)
        for j in range(T):
            V = (pos0 + j + 1) // 4
            tk[j, :min(V, 64)] = np.arange(min(V, 64))
    out = orc.attention(st, q, raw_new, tk, pos0)
    for j in range(T):
        t = pos0 + j
        rows = []
        for p in range(max(0, t - S + 1), t + 1):
            rows.append(raw_new[p - pos0] if p >= pos0 else st.raw[p % S])
        if ratio == 4:
            rows += [st.attn.comp[c] for c in range(min((t + 1) // 4, 64))]
        elif ratio == 128:
            rows += [st.attn.comp[c] for c in range((t + 1) // 128)]
        want = dense_attention(q[j], rows, shape.attn_scale)
        np.testing.assert_allclose(out[j], want, rtol=1e-6, atol=1e-7)


def test_attention_single_row_and_topk_rules(orc):
    shape, L, st, rng = _attn_state(orc, 0)
    q = rng.standard_normal((1, shape.n_heads, shape.head_dim)).astype(np.float32)
    raw_new = rng.standard_normal((1, shape.head_dim)).astype(np.float32)
    out = orc.attention(st, q, raw_new, None, 0)
    for h in range(shape.n_heads):
        np.testing.assert_allclose(out[0, h], raw_new[0], rtol=1e-7)
    # ratio 4: -1 entries are skipped, the first index >= visible ends the list
    shape, L, st, rng = _attn_state(orc, 4, k=6)
    pos0 = 40                                     # visible = 10
    q = rng.standard_normal((1, shape.n_heads, shape.head_dim)).astype(np.float32)
    raw_new = rng.standard_normal((1, shape.head_dim)).astype(np.float32)
    tk = np.array([[-1, 2, -1, 7, 10, 3]], np.int32)
    out = orc.attention(st, q, raw_new, tk, pos0)
    rows = [st.raw[p % 16] for p in range(pos0 - 15, pos0)] + [raw_new[0], st.attn.comp[2], st.attn.comp[7]]
    np.testing.assert_allclose(out[0], dense_attention(q[0], rows, shape.attn_scale), rtol=1e-6, atol=1e-7)


def test_ring_commit_and_gather_logical_order(orc):
    for ratio in (0, 4, 128):
        S, D = 16, 8
        shape = configs.LayerShape(d_model=8, head_dim=D, n_rot=4, idx_head_dim=4, n_heads=1, ratio=ratio,
                                   swa=S, top_k=2, dtype="f32")
        L = orc_layer(shape, comp_cap=64, idx_cap=64)
        st = orc.State(L)
        orc.state_init(st)
        pos = 0
        for n in (5, 9, 1, 30, 3):               # wraps the ring; ends at 48 + 0 = 48
            rows = np.stack([np.full(D, p, np.float32) for p in range(pos, pos + n)])
            orc.ring_commit(st, rows, pos)
            pos += n
        for p in range(pos - S, pos):
            assert np.all(st.raw[p % S] == p)
        for end in (pos, 3):
            if end == 3:
                st2 = orc.State(L)
                orc.state_init(st2)
                orc.ring_commit(st2, np.stack([np.full(D, p, np.float32) for p in range(3)]), 0)
                g = orc.checkpoint_gather(st2, 3)
                n_live = 3
            else:
                g = orc.checkpoint_gather(st, end)
                n_live = S
            assert g.size == orc.checkpoint_floats(L, end)
            raw_part = g[:n_live * D].reshape(n_live, D)
            np.testing.assert_array_equal(raw_part[:, 0], np.arange(end - n_live, end, dtype=np.float32))
        # closed-form size
        p = 1000
        coff = 2 if ratio == 4 else 1
        want = S * D
        if ratio:
            want += (p // ratio) * D + 2 * (coff * ratio) * (coff * D)
        if ratio == 4:
            want += (p // 4) * 4 + 2 * 8 * 8
        assert orc.checkpoint_floats(L, p) == want


@pytest.mark.parametrize("ratio", [0, 4, 128])
def test_checkpoint_restore_resumes_exactly(orc, ratio):
    """Gather at T1, restore into a fresh state, continue to T1 + T2: the state
    equals the uninterrupted run's bit for bit ([P1] §6-§7: logical-order raw
    rows and the frontier are what compression needs to continue)."""
    shape = configs.LayerShape(d_model=32, head_dim=16, n_rot=8, idx_head_dim=8, n_heads=2, ratio=ratio,
                               swa=16, top_k=4, dtype="f32", w_std=0.2)
    T1, T2 = 37, 150                                   # T1 mid-window, past the ring; T2 wraps the ring
    L = orc_layer(shape, comp_cap=64, idx_cap=64)
    wa = lane_np(configs.lane_weights(shape, 9, 0, "attn"))
    wi = lane_np(configs.lane_weights(shape, 9, 0, "idx"))
    h = np_in(configs.hidden(shape, 9, T1 + T2))
    _, _, raw = configs.queries(shape, 9, T1 + T2)
    raw = raw.numpy()

    def run(st, p0, n):
        if ratio:
            orc.compress(st, wa, wi, h[p0:p0 + n], p0)
        orc.ring_commit(st, raw[p0:p0 + n], p0)

    full = orc.State(L)
    orc.state_init(full)
    run(full, 0, T1)
    run(full, T1, T2)

    part = orc.State(L)
    orc.state_init(part)
    run(part, 0, T1)
    body = orc.checkpoint_gather(part, T1)
    fresh = orc.State(L)
    orc.state_init(fresh)
    orc.checkpoint_scatter(fresh, T1, body)
    np.testing.assert_array_equal(orc.checkpoint_gather(fresh, T1), body)
    run(fresh, T1, T2)
    np.testing.assert_array_equal(orc.checkpoint_gather(fresh, T1 + T2), orc.checkpoint_gather(full, T1 + T2))


# --------------------------------------------------------------------------
# DSV4 payload of a layer stack ("【#4】ds4.c を読み解く" §5 body order)
# --------------------------------------------------------------------------

def _payload_stack(orc, ratios, pos, S=16, D=64, d=16):
    states = []
    for li, r in enumerate(ratios):
        shape = configs.LayerShape(d_model=32, head_dim=D, n_rot=16, idx_head_dim=d, n_heads=8, ratio=r, swa=S,
                                   top_k=4, dtype="f32")
        L = orc_layer(shape, comp_cap=max(pos // max(r, 1), 1) + 3, idx_cap=pos // 4 + 3)
        st = orc.State(L)
        base = 10000.0 * (li + 1)
        # every element tells where it lives: layer, tensor, row, column
        st.raw[:] = base + 100.0 * np.arange(S)[:, None] + np.arange(D)[None, :] / 1000.0
        for k, lane in enumerate((st.attn, st.idx)):
            for j, arr in enumerate((lane.comp, lane.state_kv, lane.state_score)):
                arr[:] = base + 1000.0 * (1 + 3 * k + j) + np.arange(arr.size).reshape(arr.shape) / 64.0
        states.append(st)
    return states


def test_payload_layout_follows_the_page(orc):
    """Bytes of the oracle's DSV4 payload against the page's header table and body
    order, parsed here field by field (little-endian u32 / f32)."""
    g = _golden("payload_header.json")
    ratios, pos, S = (0, 4, 128, 4), 301, 16
    states = _payload_stack(orc, ratios, pos, S=S)
    D, d = 64, 16
    vocab = 7
    fields = dict(ctx_size=1024, prefill_chunk=4096, raw_cap=S, raw_window=S, comp_cap=200, token_count=pos,
                  layer_count=len(ratios), head_dim=D, idx_head_dim=d, vocab_size=vocab, live_raw_rows=min(pos, S))
    assert tuple(fields) == tuple(g["fields"][2:]) == orc.PAYLOAD_FIELDS
    tokens = (np.arange(pos, dtype=np.uint32) * 7919 + 3) % 128000
    logits = np.linspace(-3, 3, vocab).astype(np.float32)
    buf = orc.payload_write([fields[k] for k in orc.PAYLOAD_FIELDS], states, tokens, logits)
    u32 = buf.view("<u4")
    f32 = buf.view("<f4")
    assert buf[:4].tobytes() == g["magic_ascii"].encode() and u32[0] == g["magic_u32"]
    assert u32[1] == g["version"]
    for i, name in enumerate(g["fields"][2:], start=2):
        assert u32[i] == fields[name], name
    o = 13
    np.testing.assert_array_equal(u32[o:o + pos], tokens); o += pos                      # token ids
    np.testing.assert_array_equal(f32[o:o + vocab], logits); o += vocab                  # logits
    np.testing.assert_array_equal(u32[o:o + len(ratios)], [pos // r if r else 0 for r in ratios]); o += len(ratios)
    np.testing.assert_array_equal(u32[o:o + len(ratios)], [pos // 4 if r == 4 else 0 for r in ratios])
    o += len(ratios)
    for st, r in zip(states, ratios):
        n_live = min(pos, S)
        want = [st.raw[p % S] for p in range(pos - n_live, pos)]                        # raw rows, logical order
        if r:
            want += [st.attn.comp[:pos // r].ravel(), st.attn.state_kv.ravel(), st.attn.state_score.ravel()]
        if r == 4:
            want += [st.idx.comp[:pos // 4].ravel(), st.idx.state_kv.ravel(), st.idx.state_score.ravel()]
        w = np.concatenate([np.ravel(x) for x in want]).astype(np.float32)
        np.testing.assert_array_equal(f32[o:o + w.size], w)
        o += w.size
    assert 4 * o == buf.size


def test_payload_round_trip_restores_every_layer(orc):
    ratios, pos = (128, 4, 0, 4), 517
    states = _payload_stack(orc, ratios, pos)
    fields = [2048, 4096, 16, 16, 300, pos, len(ratios), 64, 16, 5, 16]
    tokens = np.arange(pos, dtype=np.uint32)
    logits = np.arange(5, dtype=np.float32) - 2.5
    buf = orc.payload_write(fields, states, tokens, logits)
    fresh = [orc.State(s.L) for s in states]
    f, tk, lg = orc.payload_read(buf, fresh, pos, 5)
    assert f.tolist() == fields
    np.testing.assert_array_equal(tk, tokens)
    np.testing.assert_array_equal(lg, logits)
    for a, b in zip(states, fresh):
        n_live = min(pos, a.L.swa)
        for p in range(pos - n_live, pos):
            np.testing.assert_array_equal(b.raw[p % a.L.swa], a.raw[p % a.L.swa])
        if a.L.ratio:
            np.testing.assert_array_equal(b.attn.comp[:pos // a.L.ratio], a.attn.comp[:pos // a.L.ratio])
            np.testing.assert_array_equal(b.attn.state_kv, a.attn.state_kv)
            np.testing.assert_array_equal(b.attn.state_score, a.attn.state_score)
        if a.L.ratio == 4:
            np.testing.assert_array_equal(b.idx.comp[:pos // 4], a.idx.comp[:pos // 4])
            np.testing.assert_array_equal(b.idx.state_kv, a.idx.state_kv)
            np.testing.assert_array_equal(b.idx.state_score, a.idx.state_score)
    # a corrupted magic is refused
    bad = buf.copy()
    bad[0] ^= 1
    with pytest.raises(AssertionError):
        orc.payload_read(bad, [orc.State(s.L) for s in states], pos, 5)


# --------------------------------------------------------------------------
# Full indexer: Hadamard + FP4 round trip, multi-head score
# ("Metal グラフと圧縮 KV の実装を読む" §6 and §9)
# --------------------------------------------------------------------------

def _sylvester(n):
    return np.array([[(-1) ** bin(i & j).count("1") for j in range(n)] for i in range(n)], dtype=np.float64)


def test_hadamard_sylvester_and_evaluation(orc):
    g = _golden("hadamard_sylvester.json")
    for name, n in (("H2", 2), ("H4", 4), ("H8", 8)):
        np.testing.assert_array_equal(_sylvester(n), np.array(g[name], dtype=np.float64))
    for n in (2, 8, 64, 128):
        Hm = _sylvester(n)
        np.testing.assert_array_equal(Hm @ Hm.T, n * np.eye(n))
        c = np.float32(1.0 / math.sqrt(n))
        # unit vectors: every butterfly step is exact, so column k comes out as H[:, k] * fp32(1/sqrt(n))
        for k in sorted({0, 1, min(n // 2 + 1, n - 1), n - 1}):
            e = np.zeros(n, np.float32)
            e[k] = 1.0
            np.testing.assert_array_equal(orc.hadamard(e), (Hm[:, k] * np.float64(c)).astype(np.float32))
        rng = np.random.default_rng(n)
        for _ in range(20):
            x = rng.standard_normal(n).astype(np.float32)
            y = orc.hadamard(x)
            exact = Hm @ x.astype(np.float64) / math.sqrt(n)
            # log2(n) rounded add/sub stages and one rounded multiply
            bound = (math.log2(n) + 2) * 2.0 ** -24 * np.abs(x).astype(np.float64).sum() / math.sqrt(n) * 2
            assert np.max(np.abs(y - exact)) <= bound
            np.testing.assert_allclose(np.linalg.norm(y), np.linalg.norm(x), rtol=1e-5)
            np.testing.assert_allclose(orc.hadamard(y), x, rtol=1e-5, atol=1e-5)     # orthonormal and symmetric


def test_hadamard_evaluation_order_is_the_butterfly(orc):
    """The binary32 values are those of the stage-by-stage butterfly (written out here
    independently), not of a row-by-row matrix product: the FP4 codes depend on them."""
    rng = np.random.default_rng(21)
    n = 128
    Hm = _sylvester(n)
    differs = 0
    for _ in range(50):
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3, n)).astype(np.float32)
        y = x.copy()
        h = 1
        while h < n:
            for j in range(n):
                if j & h == 0:
                    a, b = y[j], y[j + h]
                    y[j], y[j + h] = np.float32(a + b), np.float32(a - b)
            h *= 2
        y = (y * np.float32(1.0 / math.sqrt(n))).astype(np.float32)
        np.testing.assert_array_equal(orc.hadamard(x), y)
        rowwise = np.array([np.float32(np.sum((Hm[i] * x).astype(np.float32), dtype=np.float32)) for i in range(n)],
                           np.float32) * np.float32(1.0 / math.sqrt(n))
        differs += int(np.any(rowwise != y))
    assert differs > 0


def test_e2m1_format_golden(orc):
    g = _golden("e2m1_format.json")
    for v in g["values"]:
        assert orc.e2m1_rne(np.float32(v)) == v and orc.e2m1_rne(np.float32(-v)) == -v
    for y, want in g["round_cases"]:
        assert orc.e2m1_rne(np.float32(y)) == np.float32(want), y
    # brute force over a fine grid: nearest grid value, ties to the even code
    grid = np.array(g["values"])
    for y in np.linspace(0, 7, 2801):
        a = min(abs(y), 6.0)
        d = np.abs(grid - a)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
        assert orc.e2m1_rne(np.float32(y)) == np.float32(grid[code])


def test_fp4_roundtrip_properties(orc):
    rng = np.random.default_rng(23)
    g = np.array(_golden("e2m1_format.json")["values"])
    for a in np.concatenate([10.0 ** rng.uniform(-6, 6, 300), [6.0, 3.0, 12.0, 6.0000005]]):
        a = np.float32(a)
        e = orc.fp4_scale_exp(a)
        assert a <= 6.0 * 2.0 ** e and a > 6.0 * 2.0 ** (e - 1)
    assert orc.fp4_scale_exp(0.0) == 0
    x = (rng.standard_normal((5, 128)) * rng.uniform(0.01, 100, (5, 1))).astype(np.float32)
    x[2, 32:64] = 0.0
    y = orc.fp4_roundtrip(x)
    np.testing.assert_array_equal(y[2, 32:64], 0.0)
    for i in range(5):
        for b in range(4):
            blk, src = y[i, 32 * b:32 * b + 32], x[i, 32 * b:32 * b + 32]
            e = orc.fp4_scale_exp(np.max(np.abs(src)))
            mags = np.abs(blk.astype(np.float64)) * 2.0 ** -e
            assert np.all(np.isin(mags, g))                                      # on the grid
            # half a grid step: at most 0.25 * 2^e below magnitude 2^e, at most a quarter of |x| above it
            assert np.all(np.abs(blk - src) <= np.maximum(0.25 * 2.0 ** e, 0.25 * np.abs(src)))
            # each block depends on its own 32 values only
            z = x[i].copy()
            z[(32 * b + 32) % 128:(32 * b + 32) % 128 + 32] *= 3.0
            np.testing.assert_array_equal(orc.fp4_roundtrip(z)[32 * b:32 * b + 32], blk)
    np.testing.assert_array_equal(orc.fp4_roundtrip(y), y)                       # fixed points
    np.testing.assert_array_equal(orc.indexer_qat(x), orc.fp4_roundtrip(orc.hadamard(x)))


def test_index_score_heads_is_the_in_order_chain(orc):
    """Per-head fmaf chains, ReLU, and the weighted head sum as one more in-order fmaf
    chain, computed here in exact rational arithmetic."""
    from fractions import Fraction

    from fp_exact import fma_chain, round_f32
    rng = np.random.default_rng(29)
    separated = 0
    for trial in range(60):
        H, d = int(rng.integers(1, 7)), int(rng.integers(2, 9))
        q = rng.uniform(-2, 2, (H, d)).astype(np.float32)
        w = rng.uniform(-1.5, 2, H).astype(np.float32)
        row = rng.uniform(-2, 2, d).astype(np.float32)
        dots = [fma_chain(q[j], row) for j in range(H)]
        s = np.float32(0.0)
        for j in range(H):
            r = dots[j] if dots[j] > 0 else np.float32(0.0)
            s = round_f32(Fraction(float(w[j])) * Fraction(float(r)) + Fraction(float(s)))
        assert np.float32(orc.index_score_heads(q, w, row)) == s, trial
        # an unfused head sum, or no ReLU, would give another value on some of these
        u = np.float32(0.0)
        for j in range(H):
            r = dots[j] if dots[j] > 0 else np.float32(0.0)
            u = np.float32(u + np.float32(w[j] * r))
        nr = np.float32(0.0)
        for j in range(H):
            nr = round_f32(Fraction(float(w[j])) * Fraction(float(dots[j])) + Fraction(float(nr)))
        separated += int(u != s) + int(nr != s)
    assert separated > 10


def test_indexer_topk_heads_brute_force(orc):
    from compressed_kv_sparse_compressor_gb300 import configs as cf
    for qat in (0, 1):
        shape = cf.LayerShape(d_model=64, head_dim=128, n_rot=32, idx_head_dim=64, n_heads=8, ratio=4, top_k=5,
                              dtype="f32")
        L = orc_layer(shape, comp_cap=40, idx_cap=40)
        L.idx_heads, L.idx_qat = 4, qat
        st = orc.State(L)
        rng = np.random.default_rng(31 + qat)
        st.idx.comp[:] = rng.standard_normal(st.idx.comp.shape).astype(np.float32)
        pos = np.array([0, 3, 7, 19, 25, 101, 159])
        q = rng.standard_normal((len(pos), 4, 64)).astype(np.float32)
        w = rng.uniform(0.1, 1, (len(pos), 4)).astype(np.float32)
        tk, sc = orc.indexer_topk_heads(st, q, w, pos, want_scores=True)
        for j, t in enumerate(pos):
            V = (t + 1) // 4
            qj = orc.indexer_qat(q[j]) if qat else q[j]
            s = [orc.index_score_heads(qj, w[j], st.idx.comp[c]) for c in range(V)]
            want = sorted(sorted(range(V), key=lambda c: (-s[c], c))[:5])
            assert tk[j].tolist() == want + [-1] * (5 - len(want))
            np.testing.assert_array_equal(sc[j, :V], np.array(s, np.float32))
            # the score is a ReLU-weighted sum: with one head and w = 1 it is max(dot, 0)
            d0 = orc.index_score(qj[0], st.idx.comp[0]) if V else 0.0
            if V:
                np.testing.assert_equal(np.float32(orc.index_score_heads(qj[:1], np.ones(1, np.float32),
                                                                         st.idx.comp[0])), np.float32(max(d0, 0.0)))


def test_compressor_indexer_lane_qat(orc):
    """With the round trip on, every indexer row is the QAT image of the row the
    same compressor makes without it (after RMSNorm and RoPE); the attention lane
    is unchanged."""
    shape = _small_shape(4, D=128, d=64, R=32)
    wa = configs.lane_weights(shape, 3, 0, "attn")
    wi = configs.lane_weights(shape, 3, 0, "idx")
    h = configs.hidden(shape, 3, 37)
    outs = []
    for qat in (0, 1):
        L = orc_layer(shape, comp_cap=16, idx_cap=16)
        L.idx_qat = qat
        st = orc.State(L)
        orc.state_init(st)
        orc.compress(st, lane_np(wa), lane_np(wi), np_in(h), 0)
        outs.append(st)
    n = 37 // 4
    np.testing.assert_array_equal(outs[1].attn.comp[:n], outs[0].attn.comp[:n])
    np.testing.assert_array_equal(outs[1].idx.comp[:n], orc.indexer_qat(outs[0].idx.comp[:n]))
    np.testing.assert_array_equal(outs[1].idx.state_kv, outs[0].idx.state_kv)
