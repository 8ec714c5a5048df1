"""Projection GEMM (tcgen05 path for bf16, CUDA-core path for fp32) against a
float64 matmul of the same operands.  White-box: reads the projection block
the library keeps at the start of its workspace ([rows][P] float, columns
attn kv | attn score | idx kv | idx score)."""

import pytest
import torch

from compressed_kv_sparse_compressor_gb300 import configs
from gpu_util import device_layer, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("dtype,d_model,T,D,d", [
    ("bf16", 512, 300, 512, 128),      # ragged M, 2 n-tiles per kv matrix
    ("bf16", 4096, 4096, 512, 128),    # full chunk of the long-context layer (last 16 tiles split in 8 along K)
    ("bf16", 4096, 2000, 512, 128),    # 160 tiles: the last 8 split in 16 along K, ragged last m-tile
    ("bf16", 4096, 64, 512, 128),      # narrow-tile tensor-core path
    ("bf16", 4096, 32, 512, 128),      # decode batch of 32 sequences
    ("bf16", 512, 1, 512, 128),        # a single row
    ("f32", 256, 64, 128, 64),         # fp32 throughout: CUDA-core path
])
def test_projection_matches_matmul(dtype, d_model, T, D, d):
    shape = configs.LayerShape(d_model=d_model, head_dim=D, n_rot=64, idx_head_dim=d, n_heads=64, ratio=4,
                               top_k=16, dtype=dtype)
    dl, wa, wi = device_layer(shape, comp_cap=T // 4 + 1, idx_cap=T // 4 + 1, max_rows=T, seed=3)
    h = configs.hidden(shape, 3, T).cuda()
    dl.compress_prefill(h, 0)
    dl.sync()
    P = 2 * 2 * D + 2 * 2 * d
    proj = dl.ws[: T * P * 4].view(torch.float32).view(T, P)
    hd = h.double()
    want = torch.cat([hd @ w.cuda().double().T for w in (wa[0], wa[1], wi[0], wi[1])], dim=1)
    err = (proj.double() - want).abs()
    tol = 1e-4 + 2e-3 * want.abs()
    bad = (err > tol).sum().item()
    assert bad == 0, f"{bad} elements out of tolerance, max err {err.max().item():.3e}"
