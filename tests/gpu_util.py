"""Helpers of the GPU parity tests: device layers from a workload, download of a
device state into an oracle state, and the stage comparisons of the parity
protocol (each call checked against the oracle run on that call's own inputs)."""

from __future__ import annotations

import numpy as np
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs
from compressed_kv_sparse_compressor_gb300 import build as build_mod
from compressed_kv_sparse_compressor_gb300.layer import DeviceLayer
from helpers import fp8_block_exp, lane_np, np_in, orc_layer

RTOL, ATOL = 2e-3, 1e-4          # fp32-accumulated floats (spec tolerance)


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_mod.build()


def device_layer(shape, comp_cap, idx_cap=0, n_seq=1, max_rows=4096, seed=0, layer=0, gamma_std=0.0,
                 with_prequant=True):
    dl = DeviceLayer(shape, comp_cap, idx_cap, n_seq=n_seq, max_rows=max_rows, with_prequant=with_prequant)
    wa = wi = None
    if shape.ratio:
        wa = configs.lane_weights(shape, seed, layer, "attn", gamma_std=gamma_std)
    if shape.ratio == 4:
        wi = configs.lane_weights(shape, seed, layer, "idx", gamma_std=gamma_std)
    if shape.ratio:
        dl.set_weights(wa, wi)
    dl.state_init()
    return dl, wa, wi


def download(dl: DeviceLayer, b: int = 0) -> orc.State:
    """Oracle-side copy of sequence b of a device layer's state."""
    L = orc_layer(dl.shape, dl.comp_cap, dl.idx_cap)
    st = orc.State(L)
    torch.cuda.synchronize()
    st.raw[:] = dl.raw[b].cpu().numpy()
    if dl.shape.ratio:
        st.attn.comp[:] = dl.attn_comp[b].cpu().numpy()
        st.attn.state_kv[:] = dl.attn_kv[b].cpu().numpy()
        st.attn.state_score[:] = dl.attn_score[b].cpu().numpy()
        if dl.attn_pre is not None:
            st.attn.prequant[:] = dl.attn_pre[b].cpu().numpy()
    if dl.shape.ratio == 4:
        st.idx.comp[:] = dl.idx_comp[b].cpu().numpy()
        st.idx.state_kv[:] = dl.idx_kv[b].cpu().numpy()
        st.idx.state_score[:] = dl.idx_score[b].cpu().numpy()
        st.idx.prequant[:] = dl.idx_pre[b].cpu().numpy() if getattr(dl, "idx_pre", None) is not None else st.idx.comp
    return st


def clone_state(st: orc.State) -> orc.State:
    c = orc.State(st.L)
    c.raw[:] = st.raw
    for a, b in ((c.attn, st.attn), (c.idx, st.idx)):
        a.comp[:] = b.comp
        a.prequant[:] = b.prequant
        a.state_kv[:] = b.state_kv
        a.state_score[:] = b.state_score
    return c


_E4M3 = None


def _e4m3_grid():
    global _E4M3
    if _E4M3 is None:
        g = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
        _E4M3 = np.unique(g.astype(np.float64))                  # 0 .. 448, ascending
    return _E4M3


def unexplained_fp8_flips(gpu_pre, gpu_fin, orc_pre, orc_fin, n_nope):
    """FP8 elements where the GPU's row and the oracle's differ, that neither an E4M3
    rounding midpoint nor a block-scale boundary explains: each must have the oracle's
    pre-quantisation value within the pre-quantisation tolerance of a midpoint between
    two grid values (scaled by the block's 2^e), or sit in a block whose amax is within
    that tolerance of the scale boundary 448 * 2^e."""
    grid = _e4m3_grid()
    bad = 0
    for r in range(gpu_fin.shape[0]):
        for b0 in range(0, n_nope, 64):
            sl = slice(b0, min(b0 + 64, n_nope))
            diff = ~np.isclose(gpu_fin[r, sl], orc_fin[r, sl], rtol=RTOL, atol=ATOL)
            if not diff.any():
                continue
            po = orc_pre[r, sl].astype(np.float64)
            pg = gpu_pre[r, sl].astype(np.float64)
            amax_o = float(np.abs(po).max())
            e_o, e_g = fp8_block_exp(amax_o), fp8_block_exp(float(np.abs(pg).max()))
            if e_o != e_g:
                if abs(amax_o - 448.0 * 2.0 ** min(e_o, e_g)) <= ATOL + RTOL * amax_o:
                    continue
                bad += int(diff.sum())
                continue
            y = np.abs(po[diff]) * 2.0 ** -e_o
            t = (ATOL + RTOL * np.abs(po[diff])) * 2.0 ** -e_o
            i = np.searchsorted(grid, y, side="right")
            lo = grid[np.clip(i - 1, 0, len(grid) - 1)]
            hi = grid[np.clip(i, 0, len(grid) - 1)]
            near_mid = np.abs(y - (lo + hi) / 2) <= t
            # y just below a grid value can round up: the midpoint below it counts too
            lo2 = grid[np.clip(i - 2, 0, len(grid) - 1)]
            near_mid |= np.abs(y - (lo2 + lo) / 2) <= t
            bad += int((~near_mid).sum())
    return bad


def check_compress(before: orc.State, after_gpu: orc.State, wa, wi, hidden: torch.Tensor, pos0: int,
                   report=None):
    """Run the oracle's compressor from the GPU's before-state on the same hidden
    rows; compare the rows this call appended and the frontier it left."""
    L = before.L
    ref = clone_state(before)
    orc.compress(ref, lane_np(wa), lane_np(wi) if wi is not None else None, np_in(hidden), pos0)
    T = hidden.shape[0]
    r = L.ratio
    rows = slice(pos0 // r, (pos0 + T) // r)
    n_nope = L.head_dim - L.n_rot
    gp, op = after_gpu.attn.prequant[rows], ref.attn.prequant[rows]
    np.testing.assert_allclose(gp, op, rtol=RTOL, atol=ATOL, err_msg="attn pre-FP8 rows")
    gc = after_gpu.attn.comp[rows]
    # the GPU's FP8 round trip is bit-exact against the oracle's on the same input
    np.testing.assert_array_equal(orc.fp8_roundtrip(gp, n_nope), gc, err_msg="attn FP8 arithmetic")
    # the RoPE tail carries no FP8: within tolerance
    np.testing.assert_allclose(gc[:, n_nope:], ref.attn.comp[rows][:, n_nope:], rtol=RTOL, atol=ATOL)
    flips = int(np.sum(~np.isclose(gc[:, :n_nope], ref.attn.comp[rows][:, :n_nope], rtol=RTOL, atol=ATOL)))
    total = max(gc[:, :n_nope].size, 1)
    assert flips <= max(2, total // 200), f"FP8 grid flips {flips}/{total}"
    assert unexplained_fp8_flips(gp, gc, op, ref.attn.comp[rows], n_nope) == 0, "an FP8 flip no midpoint explains"
    if report is not None:
        report["fp8_flips"] = report.get("fp8_flips", 0) + flips
        report["fp8_elems"] = report.get("fp8_elems", 0) + total
    np.testing.assert_allclose(after_gpu.attn.state_kv, ref.attn.state_kv, rtol=RTOL, atol=ATOL, err_msg="attn state_kv")
    np.testing.assert_allclose(after_gpu.attn.state_score, ref.attn.state_score, rtol=RTOL, atol=ATOL,
                               err_msg="attn state_score")
    if r == 4 and L.idx_qat:
        # indexer rows with the Hadamard + FP4 round trip: the GPU's own pre-round-trip row,
        # re-quantised by the oracle, equals the GPU row bit for bit; the pre-round-trip rows
        # agree within tolerance, so an end-to-end code flip can only be a rounding straddle
        irows = slice(pos0 // 4, (pos0 + T) // 4)
        gpi = after_gpu.idx.prequant[irows]
        np.testing.assert_allclose(gpi, ref.idx.prequant[irows], rtol=RTOL, atol=ATOL, err_msg="idx pre-QAT rows")
        np.testing.assert_array_equal(orc.indexer_qat(gpi), after_gpu.idx.comp[irows], err_msg="idx QAT arithmetic")
        gi, oi = after_gpu.idx.comp[irows], ref.idx.comp[irows]
        iflips = int(np.sum(gi != oi))
        assert iflips <= max(2, gi.size // 200), f"FP4 flips {iflips}/{gi.size}"
        if report is not None:
            report["fp4_flips"] = report.get("fp4_flips", 0) + iflips
        np.testing.assert_allclose(after_gpu.idx.state_kv, ref.idx.state_kv, rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(after_gpu.idx.state_score, ref.idx.state_score, rtol=RTOL, atol=ATOL)
    elif r == 4:
        irows = slice(pos0 // 4, (pos0 + T) // 4)
        np.testing.assert_allclose(after_gpu.idx.comp[irows], ref.idx.comp[irows], rtol=RTOL, atol=ATOL,
                                   err_msg="idx rows")
        np.testing.assert_allclose(after_gpu.idx.state_kv, ref.idx.state_kv, rtol=RTOL, atol=ATOL)
        np.testing.assert_allclose(after_gpu.idx.state_score, ref.idx.state_score, rtol=RTOL, atol=ATOL)
    # rows outside this call's range are untouched
    np.testing.assert_array_equal(after_gpu.attn.comp[:pos0 // r], before.attn.comp[:pos0 // r])
    return ref


def check_split_mirror(dl, upto_rows=None):
    """The attention lane's bf16 mirror is the hi / lo split of the compressed rows, bit for bit."""
    if dl.attn_split is None:
        return
    torch.cuda.synchronize()
    comp = dl.attn_comp if upto_rows is None else dl.attn_comp[:, :upto_rows]
    split = dl.attn_split if upto_rows is None else dl.attn_split[:, :upto_rows]
    hi = comp.to(torch.bfloat16)
    lo = (comp - hi.float()).to(torch.bfloat16)
    assert torch.equal(split[:, :, 0], hi.view(torch.int16)), "mirror hi"
    assert torch.equal(split[:, :, 1], lo.view(torch.int16)), "mirror lo"


def ring_for(st: orc.State, raw_new: np.ndarray, pos0: int, t: int) -> orc.State:
    """State whose ring holds, at slot p % S, the raw row of every position
    p in [t-S+1, t-1], taking p >= pos0 from raw_new (test-side marshalling)."""
    S = st.L.swa
    s2 = orc.State.__new__(orc.State)
    s2.L, s2.attn, s2.idx = st.L, st.attn, st.idx
    s2.raw = st.raw.copy()
    for p in range(max(0, t - S + 1), t):
        if p >= pos0:
            s2.raw[p % S] = raw_new[p - pos0]
    return s2


def check_attention_sampled(st_before: orc.State, q: np.ndarray, raw_new: np.ndarray, topk, out_gpu: np.ndarray,
                            pos0: int, sample):
    """Oracle attention for sampled queries j (position pos0 + j) on the GPU's state and top-k."""
    for j in sample:
        t = pos0 + j
        s2 = ring_for(st_before, raw_new, pos0, t)
        tk = None if topk is None else topk[j:j + 1]
        ref = orc.attention(s2, q[j:j + 1], raw_new[j:j + 1], tk, t)
        np.testing.assert_allclose(out_gpu[j], ref[0], rtol=RTOL, atol=ATOL, err_msg=f"attention query {j}")


def check_indexer_sampled(st: orc.State, q_idx: np.ndarray, positions, topk_gpu, scores_gpu, sample):
    for j in sample:
        tk, sc = orc.indexer_topk(st, q_idx[j:j + 1], [positions[j]], want_scores=True)
        V = (positions[j] + 1) // 4
        if scores_gpu is not None:
            np.testing.assert_array_equal(scores_gpu[j, :V], sc[0, :V], err_msg=f"indexer scores query {j}")
        np.testing.assert_array_equal(topk_gpu[j], tk[0], err_msg=f"top-k query {j}")
