"""The benchmark's algorithmic work counts (-m "not gpu"): the numerators of
every roofline fraction the bench line reports, pinned to closed forms and to
the per-unit figures of the workload (C5: 131072 tokens, 64 heads, head_dim
512, indexer head_dim 128, top-k 512, a 128-row window), and the attention's
row count to the rows the oracle's own top-k selects."""

import numpy as np
import pytest

import bench
import oracle as orc
from compressed_kv_sparse_compressor_gb300 import configs
from helpers import lane_np, np_in, orc_layer


def test_attention_flops_closed_form():
    s = configs.C5.layer
    # a steady-state query (t >= 2047: 512 visible compressed rows, a full window) attends 640 rows
    assert bench.attn_flops_chunk(s, 4096, 1) == 4 * 64 * 512 * 640 == 83_886_080
    # the whole step: sum over t < N of min(t + 1, 128) + min(512, (t + 1) // 4)
    N = 131072
    raw = 128 * 129 // 2 + (N - 128) * 128                     # t + 1 = 1 .. 128, then 128
    # m = t + 1: floor(m / 4) summed over m = 1 .. 2047 is 4 * (1 + .. + 511); m >= 2048 gives 512
    comp = 4 * (511 * 512 // 2) + 512 * (N - 2047)
    total = sum(bench.attn_flops_chunk(s, c * 4096, 4096) for c in range(N // 4096))
    assert total == 4 * 64 * 512 * (raw + comp)
    # 10.93 TFLOP per step: below the steady-state 83.9 MFLOP/token x 131072 = 11.0 TFLOP, since the
    # first 2047 queries see fewer than 512 compressed rows and the first 127 a partial window
    assert total == 10_925_264_338_944 < 83_886_080 * N


def test_indexer_flops_closed_form():
    s = configs.C5.layer
    N = 131072
    # sum of floor(m / 4) for m = 1 .. N (N a multiple of 4) = (N/4) * (N/2 - 1)
    vis = (N // 4) * (N // 2 - 1)
    assert vis == 2_147_450_880
    total = sum(bench.indexer_flops_chunk(s, c * 4096, 4096) for c in range(N // 4096))
    assert total == 2 * 128 * vis == 549_747_425_280          # 5.5e11 flop per step


def test_projection_and_compressor_units():
    s = configs.C5.layer
    # projection: kv and score of both lanes, 2 * coff * D + 4 * d columns of d_model
    br = {"compress_projection": 1.0, "compress_fused_pool": 1.0}

    class PF:
        shape, T, chunk, n_chunks = s, 4096, 4096, 1
    r = bench.roofline("compress", br, PF, {"bf16_tflops": 1.0, "hbm_gbs": 1.0}, "test")
    assert r["achieved"] == round(2 * 4096 * 2560 * 4096 / 1e-3 / 1e12, 2)   # 20.97 MFLOP per token
    c = bench.roofline("compressor", br, PF, {"bf16_tflops": 1.0, "hbm_gbs": 1.0}, "test")
    # read: kv and score of both lanes (2 x 2 x 512 + 2 x 2 x 128 floats); write: one fp32 row and its
    # bf16 hi/lo mirror per 4 tokens (attention lane) and one fp32 indexer row per 4 tokens
    assert c["bytes_per_token"] == 10_240 + 1_152 == 11_392


def test_attention_rows_match_the_oracle_selection():
    """attn_flops_chunk counts, per query, the window rows plus min(k, visible) compressed
    rows: the oracle's top-k on a small ratio-4 layer selects exactly that many."""
    shape = configs.LayerShape(d_model=64, head_dim=64, n_rot=16, idx_head_dim=32, n_heads=8, ratio=4, swa=16,
                               top_k=6, dtype="f32", w_std=0.1)
    T, seed = 80, 3
    st = orc.State(orc_layer(shape, T // 4 + 1, T // 4 + 1))
    orc.state_init(st)
    wa = configs.lane_weights(shape, seed, 0, "attn")
    wi = configs.lane_weights(shape, seed, 0, "idx")
    orc.compress(st, lane_np(wa), lane_np(wi), np_in(configs.hidden(shape, seed, T)), 0)
    _, q_idx, _ = configs.queries(shape, seed, T)
    tk = orc.indexer_topk(st, q_idx.numpy(), np.arange(T))
    rows = 0
    for t in range(T):
        vis = (t + 1) // 4
        sel = [i for i in tk[t] if 0 <= i < vis]
        assert len(sel) == min(shape.top_k, vis)
        rows += min(t + 1, shape.swa) + len(sel)
    assert bench.attn_flops_chunk(shape, 0, T) == 4 * shape.n_heads * shape.head_dim * rows
