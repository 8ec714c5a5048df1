"""The allocation-free indexer call against the regular one (-m gpu).

ds4c_indexer_topk_noalloc serves callers that cannot allocate device memory
(no cudaMalloc, no workspace): it keeps its score matrix in a fixed device
array inside the library.  Its top-k lists must equal those of
ds4c_indexer_topk (integer output: bit for bit) on two calls in a row, for a
decode step and for a short prefill chunk.  This file is collected last.
"""

import numpy as np
import pytest
import torch

from compressed_kv_sparse_compressor_gb300 import abi, configs
from gpu_util import device_layer, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _noalloc(dl, q_idx, positions, n_seq, n_tok, topk):
    st = abi.ds4c_indexer_topk_noalloc(dl.cfg, dl.state, q_idx.data_ptr(), abi.u64_array(positions), n_seq, n_tok,
                                       topk.data_ptr(), torch.cuda.current_stream().cuda_stream)
    abi.check(st, "ds4c_indexer_topk_noalloc")


def test_noalloc_matches_workspace_call():
    shape = configs.LayerShape(d_model=512, head_dim=512, n_rot=64, idx_head_dim=128, n_heads=64, ratio=4,
                               top_k=64, dtype="bf16", w_std=0.04)
    B, cap = 8, 2048
    dl, _, _ = device_layer(shape, comp_cap=cap, idx_cap=cap, n_seq=B, max_rows=1024, seed=41)
    g = torch.Generator(device="cuda").manual_seed(41)
    dl.idx_comp.copy_(torch.randn(dl.idx_comp.shape, generator=g, device="cuda"))
    for call in range(2):
        # decode step: one query per sequence at staggered positions
        lens = [4000 + 3 * b + call for b in range(B)]
        q = torch.randn(B, shape.idx_head_dim, generator=g, device="cuda")
        want = torch.empty(B, shape.top_k, dtype=torch.int32, device="cuda")
        got = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
        dl.indexer_topk(q, lens, B, 1, want)
        _noalloc(dl, q, lens, B, 1, got)
        dl.sync()
        assert torch.equal(got, want), f"decode call {call}"
        # prefill chunk of one sequence (the state's first sequence)
        dl0 = dl.seq_view(0)
        T, pos0 = 512, 6000 + 100 * call
        qp = torch.randn(T, shape.idx_head_dim, generator=g, device="cuda")
        want = torch.empty(T, shape.top_k, dtype=torch.int32, device="cuda")
        got = torch.full((T, shape.top_k), -7, dtype=torch.int32, device="cuda")
        saved = dl.state
        dl.state = dl0
        dl.indexer_topk(qp, [pos0], 1, T, want)
        st = abi.ds4c_indexer_topk_noalloc(dl.cfg, dl0, qp.data_ptr(), abi.u64_array([pos0]), 1, T, got.data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
        dl.state = saved
        abi.check(st, "ds4c_indexer_topk_noalloc")
        dl.sync()
        assert torch.equal(got, want), f"prefill call {call}"


def _limit_layer(n_seq, cap):
    shape = configs.LayerShape(d_model=256, head_dim=128, n_rot=64, idx_head_dim=64, n_heads=8, ratio=4, top_k=512,
                               dtype="f32")
    dl, _, _ = device_layer(shape, comp_cap=16, idx_cap=cap, n_seq=n_seq, max_rows=64, seed=43, with_prequant=False)
    g = torch.Generator(device="cuda").manual_seed(43)
    dl.idx_comp.copy_(torch.randn(dl.idx_comp.shape, generator=g, device="cuda"))
    return shape, dl, g


def test_noalloc_at_the_capacity_limit():
    """A request whose padded score matrix is exactly DS4C_NOALLOC_SCORE_FLOATS is
    served (and equals the workspace call); one padded row width more is refused."""
    lim = abi.NOALLOC_SCORE_FLOATS
    B, V = 64, 32768
    assert B * V == lim
    shape, dl, g = _limit_layer(B, V + 8)
    stream = torch.cuda.current_stream().cuda_stream
    # decode: one sequence sees V rows (the widest row sets the padded width), some see none (pos < 3)
    lens = [4 * V - 1] + [4 * (V - 37 * b) + b % 4 for b in range(1, B - 3)] + [0, 1, 2]
    q = torch.randn(B, shape.idx_head_dim, generator=g, device="cuda")
    for call in range(2):
        want = torch.empty(B, shape.top_k, dtype=torch.int32, device="cuda")
        got = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
        dl.indexer_topk(q, lens, B, 1, want)
        _noalloc(dl, q, lens, B, 1, got)
        dl.sync()
        assert torch.equal(got, want), f"decode at the limit, call {call}"
        assert (got[-3:] == -1).all()
    # one padded width (4 rows) more for the widest sequence: refused, nothing launched
    over = [4 * (V + 4) - 1] + lens[1:]
    got = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
    st = abi.ds4c_indexer_topk_noalloc(dl.cfg, dl.state, q.data_ptr(), abi.u64_array(over), B, 1, got.data_ptr(),
                                       stream)
    assert st == abi.DS4C_ERR_CAPACITY
    dl.sync()
    assert (got == -7).all()
    # prefill: 64 queries of one sequence whose last query sees V rows
    dl0 = dl.seq_view(0)
    T = B
    pos0 = 4 * V - T
    qp = torch.randn(T, shape.idx_head_dim, generator=g, device="cuda")
    want = torch.empty(T, shape.top_k, dtype=torch.int32, device="cuda")
    got = torch.full((T, shape.top_k), -7, dtype=torch.int32, device="cuda")
    saved = dl.state
    dl.state = dl0
    dl.indexer_topk(qp, [pos0], 1, T, want)
    dl.state = saved
    abi.check(abi.ds4c_indexer_topk_noalloc(dl.cfg, dl0, qp.data_ptr(), abi.u64_array([pos0]), 1, T, got.data_ptr(),
                                            stream), "ds4c_indexer_topk_noalloc")
    dl.sync()
    assert torch.equal(got, want), "prefill at the limit"
    st = abi.ds4c_indexer_topk_noalloc(dl.cfg, dl0, qp.data_ptr(), abi.u64_array([pos0 + 4]), 1, T, got.data_ptr(),
                                       stream)
    assert st == abi.DS4C_ERR_CAPACITY


def test_noalloc_rejects_oversize():
    shape = configs.C5.layer
    dl, _, _ = device_layer(shape, comp_cap=32768, idx_cap=32768, max_rows=16, seed=5, with_prequant=False)
    q = torch.zeros(4096, shape.idx_head_dim, device="cuda")
    topk = torch.empty(4096, shape.top_k, dtype=torch.int32, device="cuda")
    st = abi.ds4c_indexer_topk_noalloc(dl.cfg, dl.state, q.data_ptr(), abi.u64_array([126976]), 1, 4096,
                                       topk.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == abi.DS4C_ERR_CAPACITY
    assert 4096 * 32768 > abi.NOALLOC_SCORE_FLOATS
