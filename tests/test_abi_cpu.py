"""Host-side checks of libds4c that need no GPU: the library loads, exports every
symbol include/ds4c.h declares, sizes its buffers as the oracle does, and
rejects bad arguments on the host before anything is launched."""

import ctypes as C
import os
import re

import numpy as np
import pytest

from compressed_kv_sparse_compressor_gb300 import abi, configs
from compressed_kv_sparse_compressor_gb300 import build as build_mod
from helpers import orc_layer

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return abi.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "ds4c.h")).read()
    return sorted(set(re.findall(r"\b(ds4c_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    syms = declared_symbols()
    assert set(syms) == set(abi.EXPORTS)
    for s in syms:
        assert hasattr(L, s), s


def _cfg(shape, comp_cap=64, idx_cap=64):
    return abi.LayerCfg(d_model=shape.d_model, head_dim=shape.head_dim, n_rot=shape.n_rot,
                        idx_head_dim=shape.idx_head_dim, n_heads=shape.n_heads, ratio=shape.ratio, swa=shape.swa,
                        top_k=shape.top_k, comp_cap=comp_cap, idx_cap=idx_cap,
                        dtype=abi.DS4C_F32 if shape.dtype == "f32" else abi.DS4C_BF16, rms_eps=shape.rms_eps,
                        attn_scale=shape.attn_scale, rope_base=shape.rope_base)


def test_checkpoint_floats_matches_oracle(L, orc):
    for w in (configs.C1, configs.C2, configs.C5):
        for ratio in (0, 4, 128):
            shape = configs.LayerShape(**{**w.layer.__dict__, "ratio": ratio})
            cap = 40000
            cfg = _cfg(shape, cap, cap)
            for pos in (0, 3, 127, 128, 1000, 131072):
                assert abi.ds4c_checkpoint_floats(cfg, pos) == orc.checkpoint_floats(orc_layer(shape, cap, cap), pos)


def test_invalid_configs_are_rejected(L):
    base = configs.C1.layer
    assert abi.ds4c_workspace_bytes(_cfg(base), 64) > 0
    big = _cfg(configs.C5.layer, 32768, 32768)
    assert abi.ds4c_attn_uses_tensor_cores(big) == 1
    # fewer than 64 heads are padded to the MMA tile; more than 64 run as groups of 64
    assert abi.ds4c_attn_uses_tensor_cores(_cfg(base)) == (1 if base.head_dim in (128, 256, 512) else 0)
    many = _cfg(configs.LayerShape(**{**configs.C5.layer.__dict__, "n_heads": 128, "head_dim": 256}), 32768, 32768)
    assert abi.ds4c_attn_uses_tensor_cores(many) == 1
    # (128 heads of 512 exceed the configuration's 32768-float query row)
    too_many = _cfg(configs.LayerShape(**{**configs.C5.layer.__dict__, "n_heads": 128}), 32768, 32768)
    assert abi.ds4c_attn_uses_tensor_cores(too_many) == 0
    # a raw window of at most one 128-row tile runs on the tensor cores (shorter ones masked); longer on
    # the CUDA cores
    for swa, tc in ((32, 1), (100, 1), (128, 1), (256, 0)):
        ring = _cfg(configs.LayerShape(**{**configs.C5.layer.__dict__, "swa": swa}), 32768, 32768)
        assert abi.ds4c_attn_uses_tensor_cores(ring) == tc, swa
    # the tensor-core path holds a row list of at most 512 entries; larger top-k runs on the CUDA cores
    wide = _cfg(configs.LayerShape(**{**configs.C5.layer.__dict__, "top_k": 1024}), 32768, 32768)
    assert abi.ds4c_attn_uses_tensor_cores(wide) == 0
    assert abi.ds4c_workspace_bytes(big, 4096, 32) >= abi.ds4c_workspace_bytes(big, 4096)
    for bad in (dict(ratio=3), dict(head_dim=96), dict(n_heads=12), dict(n_rot=6), dict(d_model=100),
                dict(idx_head_dim=48), dict(swa=0), dict(top_k=0)):
        shape = configs.LayerShape(**{**base.__dict__, **bad})
        assert abi.ds4c_workspace_bytes(_cfg(shape), 64) == 0, bad


FAKE = 1 << 20          # an aligned non-NULL address that is never dereferenced


def _state():
    lane = abi.LaneState(FAKE, FAKE, FAKE, None, FAKE)
    return abi.LayerState(FAKE, lane, lane)


def _weights():
    return abi.LaneWeights(FAKE, FAKE, FAKE, None)


def test_host_validation_errors(L):
    shape = configs.C1.layer
    cfg = _cfg(shape, comp_cap=16, idx_cap=16)
    st, w = _state(), _weights()
    ws_need = abi.ds4c_workspace_bytes(cfg, 64)
    pos1 = abi.u64_array([0])
    # NULL hidden / weights
    assert abi.ds4c_compress_prefill(cfg, w, w, st, None, 64, 0, FAKE, ws_need, None) == abi.DS4C_ERR_NULL
    assert abi.ds4c_compress_prefill(cfg, None, w, st, FAKE, 64, 0, FAKE, ws_need, None) == abi.DS4C_ERR_NULL
    # ratio-4 needs the indexer lane
    assert abi.ds4c_compress_prefill(cfg, w, None, st, FAKE, 64, 0, FAKE, ws_need, None) == abi.DS4C_ERR_NULL
    # capacity: 68 tokens make 17 rows > comp_cap 16
    assert abi.ds4c_compress_prefill(cfg, w, w, st, FAKE, 68, 0, FAKE, ws_need, None) == abi.DS4C_ERR_CAPACITY
    # workspace
    assert abi.ds4c_compress_prefill(cfg, w, w, st, FAKE, 64, 0, FAKE, ws_need - 1, None) == abi.DS4C_ERR_WORKSPACE
    assert abi.ds4c_compress_prefill(cfg, w, w, st, FAKE, 64, 0, None, ws_need, None) == abi.DS4C_ERR_WORKSPACE
    # misaligned pointer
    assert abi.ds4c_compress_prefill(cfg, w, w, st, FAKE + 4, 64, 0, FAKE, ws_need, None) == abi.DS4C_ERR_SHAPE
    # n_seq > 1 with n_tok > 1
    pos2 = abi.u64_array([0, 0])
    assert abi.ds4c_indexer_topk(cfg, st, FAKE, pos2, 2, 4, FAKE, None, 0, FAKE, ws_need, None) == abi.DS4C_ERR_UNSUPPORTED
    assert abi.ds4c_sparse_swa_attn(cfg, st, FAKE, FAKE, FAKE, pos2, 2, 4, FAKE, 1, FAKE, ws_need, None) == \
        abi.DS4C_ERR_UNSUPPORTED
    # indexer on a non-ratio-4 layer
    cfg128 = _cfg(configs.LayerShape(**{**shape.__dict__, "ratio": 128}), comp_cap=16)
    assert abi.ds4c_indexer_topk(cfg128, st, FAKE, pos1, 1, 4, FAKE, None, 0, FAKE, ws_need, None) == abi.DS4C_ERR_SHAPE
    # scores buffer too narrow: 64 queries from 0 see up to 16 rows
    assert abi.ds4c_indexer_topk(cfg, st, FAKE, pos1, 1, 64, FAKE, FAKE, 15, FAKE, ws_need, None) == abi.DS4C_ERR_CAPACITY
    # ratio-4 attention needs a top-k list
    assert abi.ds4c_sparse_swa_attn(cfg, st, FAKE, FAKE, None, pos1, 1, 4, FAKE, 1, FAKE, ws_need, None) == \
        abi.DS4C_ERR_NULL
    # decode batch above the limit
    big = abi.u64_array([0] * 1025)
    assert abi.ds4c_compress_decode_step(cfg, w, w, st, FAKE, big, 1025, FAKE, ws_need, None) == \
        abi.DS4C_ERR_UNSUPPORTED
    # checkpoint buffer too small
    n = abi.ds4c_checkpoint_floats(cfg, 40)
    written = C.c_size_t(0)
    assert abi.ds4c_checkpoint_gather(cfg, st, 0, 40, FAKE, n - 1, C.byref(written), None) == abi.DS4C_ERR_CAPACITY
    assert abi.status_string(abi.DS4C_ERR_CAPACITY).startswith("positions")
    # the FMA-rate probe validates before launching
    assert abi.ds4c_fma_probe(8, 16, None, None)[0] == abi.DS4C_ERR_NULL
    assert abi.ds4c_fma_probe(0, 16, FAKE, None)[0] == abi.DS4C_ERR_SHAPE
    assert abi.ds4c_fma_probe(8, 0, FAKE, None)[0] == abi.DS4C_ERR_SHAPE
    assert abi.ds4c_fma_probe(8, (1 << 24) + 1, FAKE, None)[0] == abi.DS4C_ERR_SHAPE
    assert abi.ds4c_fma_probe(8, 16, FAKE + 2, None)[0] == abi.DS4C_ERR_SHAPE


def test_payload_header_matches_the_page_table():
    """ds4c_payload_header writes the 13 fields in the order of the page's table."""
    import json
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "payload_header.json")))
    info = abi.PayloadInfo(*range(101, 112))      # distinct values: ctx_size = 101 .. live_raw_rows = 111
    hdr = abi.ds4c_payload_header(info)
    assert len(hdr) == g["u32_fields"] == abi.PAYLOAD_U32_FIELDS
    assert hdr[0] == g["magic_u32"] == int.from_bytes(g["magic_ascii"].encode(), "little")
    assert hdr[1] == g["version"]
    names = [f[0] for f in abi.PayloadInfo._fields_]
    for i, name in enumerate(g["fields"][2:], start=2):
        assert hdr[i] == getattr(info, name), name
    assert names == g["fields"][2:]


def test_noalloc_capacity_constant_matches_the_header():
    """The binding's copy of DS4C_NOALLOC_SCORE_FLOATS is the header's value."""
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "ds4c.h")).read()
    m = re.search(r"#define\s+DS4C_NOALLOC_SCORE_FLOATS\s+\((\d+)u\s*\*\s*(\d+)u\s*\*\s*(\d+)u\)", hdr)
    assert m, "DS4C_NOALLOC_SCORE_FLOATS not found in include/ds4c.h"
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == abi.NOALLOC_SCORE_FLOATS


def test_payload_bytes_and_host_validation(L, orc):
    """ds4c_payload_bytes matches the oracle's payload size; ds4c_payload_write / read
    reject bad arguments on the host before touching the device."""
    shapes = [configs.LayerShape(d_model=64, head_dim=128, n_rot=64, idx_head_dim=64, n_heads=8, ratio=r, top_k=8,
                                 dtype="f32") for r in (0, 4, 128, 4)]
    pos, vocab = 1000, 11
    cfgs = []
    for s in shapes:
        cfgs.append(abi.LayerCfg(d_model=s.d_model, head_dim=s.head_dim, n_rot=s.n_rot, idx_head_dim=s.idx_head_dim,
                                 n_heads=s.n_heads, ratio=s.ratio, swa=s.swa, top_k=s.top_k, comp_cap=300,
                                 idx_cap=300, dtype=abi.DS4C_F32, rms_eps=s.rms_eps, attn_scale=s.attn_scale,
                                 rope_base=s.rope_base))
    states = [orc.State(orc_layer(s, comp_cap=300, idx_cap=300)) for s in shapes]
    fields = [4096, 4096, 128, 128, 300, pos, 4, 128, 64, vocab, 128]
    assert abi.ds4c_payload_bytes(cfgs, pos, vocab) == orc.payload_size(states, fields)
    assert abi.ds4c_payload_bytes(cfgs[:0] + [abi.LayerCfg()], pos, vocab) == 0
    info = abi.PayloadInfo(*fields)
    st = [abi.LayerState() for _ in cfgs]
    FAKE = 1 << 20
    tok = np.zeros(pos, np.uint32)
    lg = np.zeros(vocab, np.float32)
    need = abi.ds4c_payload_bytes(cfgs, pos, vocab)
    assert abi.ds4c_payload_write(info, cfgs, st, 0, tok, lg, None, need, None)[0] == abi.DS4C_ERR_NULL
    assert abi.ds4c_payload_write(info, cfgs, st, 0, None, lg, FAKE, need, None)[0] == abi.DS4C_ERR_NULL
    bad = abi.PayloadInfo(*fields)
    bad.layer_count = 3
    assert abi.ds4c_payload_write(bad, cfgs, st, 0, tok, lg, FAKE, need, None)[0] == abi.DS4C_ERR_SHAPE
    bad = abi.PayloadInfo(*fields)
    bad.head_dim = 256
    assert abi.ds4c_payload_write(bad, cfgs, st, 0, tok, lg, FAKE, need, None)[0] == abi.DS4C_ERR_SHAPE
    bad = abi.PayloadInfo(*fields)
    bad.live_raw_rows = 127
    assert abi.ds4c_payload_write(bad, cfgs, st, 0, tok, lg, FAKE, need, None)[0] == abi.DS4C_ERR_SHAPE
    bad = abi.PayloadInfo(*fields)
    bad.comp_cap = 299                               # a layer holds more rows than the header's capacity
    assert abi.ds4c_payload_write(bad, cfgs, st, 0, tok, lg, FAKE, need, None)[0] == abi.DS4C_ERR_SHAPE
    assert abi.ds4c_payload_write(info, cfgs, st, 0, tok, lg, FAKE + 4, need, None)[0] == abi.DS4C_ERR_SHAPE
    assert abi.ds4c_payload_write(info, cfgs, st, 0, tok, lg, FAKE, need - 1, None)[0] == abi.DS4C_ERR_CAPACITY
    big = abi.PayloadInfo(*fields)
    big.token_count, big.live_raw_rows = 1300, 128   # 1300 / 4 = 325 rows > idx_cap 300
    assert abi.ds4c_payload_write(big, cfgs, st, 0, np.zeros(1300, np.uint32), lg, FAKE, 1 << 30,
                                  None)[0] == abi.DS4C_ERR_CAPACITY
    assert abi.ds4c_payload_read(info, cfgs, st, 0, None, need, tok, lg, None)[0] == abi.DS4C_ERR_NULL
    assert abi.ds4c_payload_read(info, cfgs, st, 0, FAKE + 4, need, tok, lg, None)[0] == abi.DS4C_ERR_SHAPE
    assert abi.ds4c_payload_read(info, cfgs, st, 0, FAKE, 10, tok, lg, None)[0] == abi.DS4C_ERR_CAPACITY


def test_missing_library_fails_loudly(monkeypatch):
    """No fallback: with the shared library absent, the binding raises instead of computing."""
    monkeypatch.setattr(abi, "_lib", None)
    monkeypatch.setattr(abi, "LIB_PATH", "/nonexistent/libds4c.so")
    with pytest.raises(RuntimeError, match="not built"):
        abi.lib()
    with pytest.raises(RuntimeError):
        abi.ds4c_workspace_bytes(abi.LayerCfg(), 64)
