"""Failure detection on the GPU, in the form that faults and hangs nothing (-m gpu).

Every spin-wait in the kernels is bounded; when its limit runs out the kernel raises
a sticky device error word, drains what it still has in flight and returns.  Here a
one-CTA self-test waits on an mbarrier that nothing arrives on, so its short limit
runs out: ds4c_sync_status must report DS4C_ERR_DEVICE once, clear the word, and the
next regular call must pass parity.  A second test runs the real TMA-staged decode
score with a limit of a few nanoseconds (its waits give up or not, depending on how
fast the boxes land) and checks that either way the status path and the following
default-limit call are correct."""

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import abi, configs
from gpu_util import check_indexer_sampled, device_layer, download, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    orc.build()
    yield
    abi.check(abi.ds4c_test_set_wait_limit(0), "ds4c_test_set_wait_limit")


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _decode_indexer(seed):
    shape = configs.LayerShape(d_model=256, head_dim=128, n_rot=64, idx_head_dim=128, n_heads=8, ratio=4, top_k=64,
                               dtype="f32")
    B, cap = 16, 3000
    dl, _, _ = device_layer(shape, comp_cap=16, idx_cap=cap, n_seq=B, seed=seed, max_rows=64)
    g = torch.Generator(device="cuda").manual_seed(seed)
    dl.idx_comp.copy_(torch.randn(dl.idx_comp.shape, generator=g, device="cuda"))
    lens = [4 * cap - 1 - 37 * b for b in range(B)]
    q = torch.randn(B, shape.idx_head_dim, generator=g, device="cuda")
    return shape, dl, lens, q


def _checked_call(dl, shape, lens, q):
    B = len(lens)
    vmax = max((p + 1) // 4 for p in lens)
    topk = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((B, vmax), float("nan"), device="cuda")
    dl.indexer_topk(q, lens, B, 1, topk, scores, vmax)
    dl.sync()
    for b in (0, B // 2, B - 1):
        check_indexer_sampled(download(dl, b), q[b:b + 1].cpu().numpy(), [lens[b]], topk[b:b + 1].cpu().numpy(),
                              scores[b:b + 1].cpu().numpy(), [0])


def test_wait_that_runs_out_raises_the_error_word_once():
    st = abi.ds4c_test_wait_timeout(2000, _stream())             # 2 us on a barrier nothing arrives on
    assert st == abi.DS4C_OK
    assert abi.ds4c_sync_status(_stream()) == abi.DS4C_ERR_DEVICE
    assert abi.ds4c_sync_status(_stream()) == abi.DS4C_OK        # read and cleared
    # the context is usable and a regular call is correct
    shape, dl, lens, q = _decode_indexer(61)
    _checked_call(dl, shape, lens, q)
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 1023 * 1024 / 2


def test_short_wait_limit_on_the_decode_score():
    shape, dl, lens, q = _decode_indexer(62)
    B = len(lens)
    vmax = max((p + 1) // 4 for p in lens)
    topk = torch.full((B, shape.top_k), -7, dtype=torch.int32, device="cuda")
    scores = torch.zeros((B, vmax), device="cuda")
    assert abi.ds4c_test_set_wait_limit(5) == abi.DS4C_OK
    try:
        st = abi.ds4c_indexer_topk(dl.cfg, dl.state, q.data_ptr(), abi.u64_array(lens), B, 1, topk.data_ptr(),
                                   scores.data_ptr(), vmax, dl.ws.data_ptr(), dl.ws_bytes, _stream())
        assert st == abi.DS4C_OK
        first = abi.ds4c_sync_status(_stream())
    finally:
        assert abi.ds4c_test_set_wait_limit(0) == abi.DS4C_OK
    assert first in (abi.DS4C_OK, abi.DS4C_ERR_DEVICE)
    assert abi.ds4c_sync_status(_stream()) == abi.DS4C_OK
    # with the default limit again, the same call is correct
    _checked_call(dl, shape, lens, q)
