"""Layer stacks on the GPU (-m gpu): the Pro variant's layer table run through the
library, and the DSV4 payload of a whole stack -- written bit for bit as the oracle
writes it, read back into fresh layers, and resumed exactly."""

import numpy as np
import pytest
import torch

import oracle as orc
from compressed_kv_sparse_compressor_gb300 import abi, configs
from compressed_kv_sparse_compressor_gb300.layer import DeviceLayer
from compressed_kv_sparse_compressor_gb300 import synth
from gpu_util import (check_attention_sampled, check_compress, check_indexer_sampled, check_split_mirror,
                      device_layer, download, require_gpu)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()
    orc.build()


def _run_chunk(dl, shape, seed, p0, n, layer):
    dev = "cuda"
    h = configs.hidden(shape, seed, n, offset_tok=p0, device=dev, layer=layer)
    q, q_idx, raw = configs.queries(shape, seed, n, offset_tok=p0, device=dev, layer=layer)
    dl.compress_prefill(h, p0)
    tk = None
    if shape.ratio == 4:
        tk = torch.empty(n, shape.top_k, dtype=torch.int32, device=dev)
        dl.indexer_topk(q_idx, [p0], 1, n, tk)
    out = torch.empty(n, shape.n_heads, shape.head_dim, device=dev)
    dl.attention(q, raw, tk, [p0], 1, n, out, commit_ring=True)
    return tk, out


def test_pro_stack():
    """Pro-variant stack (layers 0-1 at ratio 128): every layer runs; the last chunk
    of layer 0 (a Pro-only ratio-128 first layer) and of the first ratio-4 layer is
    checked stage-wise against the oracle, with the checkpoint gather bit for bit."""
    w = configs.PRO
    assert list(w.ratios) == [orc.layer_ratio(1, i) for i in range(8)]
    T, C = w.n_tok, w.chunk
    rng = np.random.default_rng(6)
    checked = set()
    for li, shape in enumerate(w.layers()):
        r = shape.ratio
        dl, wa, wi = device_layer(shape, comp_cap=T // r, idx_cap=T // 4 if r == 4 else 0, seed=w.seed, layer=li,
                                  max_rows=C, with_prequant=True)
        check = li == 0 or (r == 4 and 4 not in checked)
        for c in range(T // C - (1 if check else 0)):
            _run_chunk(dl, shape, w.seed, c * C, C, li)
        if check:
            p0 = T - C
            dev = "cuda"
            h = configs.hidden(shape, w.seed, C, offset_tok=p0, device=dev, layer=li)
            q, q_idx, raw = configs.queries(shape, w.seed, C, offset_tok=p0, device=dev, layer=li)
            before = download(dl)
            dl.compress_prefill(h, p0)
            after = download(dl)
            check_compress(before, after, wa, wi, h.cpu(), p0)
            check_split_mirror(dl)
            sample = sorted(set([0, C - 1] + rng.integers(0, C, 6).tolist()))
            tk = None
            if r == 4:
                vis = (p0 + C) // 4
                tk = torch.empty(C, shape.top_k, dtype=torch.int32, device=dev)
                sc = torch.empty(C, vis, device=dev)
                dl.indexer_topk(q_idx, [p0], 1, C, tk, sc, vis)
                torch.cuda.synchronize()
                rows = np.asarray(sample)
                check_indexer_sampled(after, q_idx[rows].cpu().numpy(), [p0 + j for j in sample],
                                      tk[rows].cpu().numpy(), sc[rows].cpu().numpy(), range(len(sample)))
            out = torch.empty(C, shape.n_heads, shape.head_dim, device=dev)
            dl.attention(q, raw, tk, [p0], 1, C, out, commit_ring=True)
            dl.sync()
            check_attention_sampled(after, q.cpu().numpy(), raw.cpu().numpy(),
                                    None if tk is None else tk.cpu().numpy(), out.cpu().numpy(), p0, sample)
            n = dl.checkpoint_floats(T)
            dst = torch.empty(n, device="cuda")
            assert dl.checkpoint_gather(0, T, dst) == n
            dl.sync()
            np.testing.assert_array_equal(dst.cpu().numpy(), orc.checkpoint_gather(download(dl), T))
            checked.add(r if li else "first")
        dl.sync()
        del dl
        torch.cuda.empty_cache()
    assert checked == {"first", 4}


def _stack(w, T_cap, layers):
    out = []
    for li, shape in enumerate(w.layers()[:layers]):
        r = shape.ratio
        dl, wa, wi = device_layer(shape, comp_cap=max(T_cap // max(r, 1), 1), idx_cap=T_cap // 4 if r == 4 else 0,
                                  seed=w.seed, layer=li, max_rows=4096, with_prequant=False)
        out.append((shape, dl, wa, wi))
    return out


def _fresh_like(shape, dl, wa, wi):
    d2 = DeviceLayer(shape, dl.comp_cap, dl.idx_cap, n_seq=1, max_rows=4096, with_prequant=False)
    if shape.ratio:
        d2.set_weights(wa, wi)
    d2.state_init()
    return d2


def _tensors(dl):
    return [t for t in (dl.raw, dl.attn_comp, dl.attn_kv, dl.attn_score, dl.attn_split, dl.idx_comp, dl.idx_kv,
                        dl.idx_score) if t is not None]


def test_payload_of_the_flash_stack_is_bit_exact_and_resumes():
    """The C3 stack's eight layers after 5157 tokens (the ring wrapped, frontiers mid-window):
    the GPU payload equals the oracle's payload of the downloaded states byte for byte;
    read back into fresh layers, one more 523-token chunk gives the same outputs and states,
    bit for bit, as the uninterrupted stack."""
    w = configs.C3
    pos, more = 4096 + 1061, 523
    stack = _stack(w, pos + more, 8)
    for li, (shape, dl, _, _) in enumerate(stack):
        _run_chunk(dl, shape, w.seed, 0, 4096, li)
        _run_chunk(dl, shape, w.seed, 4096, pos - 4096, li)
        dl.sync()
    vocab = 1000
    tokens = (synth.normal(w.seed, 900, (pos,)).abs() * 1e4).to(torch.int64).numpy().astype(np.uint32)
    logits = synth.normal(w.seed, 901, (vocab,)).numpy()
    D, d = w.layer.head_dim, w.layer.idx_head_dim
    fields = [pos + more, 4096, 128, 128, max(dl.comp_cap for _, dl, _, _ in stack), pos, 8, D, d, vocab, 128]
    info = abi.PayloadInfo(*fields)
    cfgs = [dl.cfg for _, dl, _, _ in stack]
    states = [dl.state for _, dl, _, _ in stack]
    nbytes = abi.ds4c_payload_bytes(cfgs, pos, vocab)
    buf = torch.full((nbytes + 64,), 0xAB, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    s, written = abi.ds4c_payload_write(info, cfgs, states, 0, tokens, logits, buf.data_ptr(), buf.numel(), stream)
    abi.check(s, "ds4c_payload_write")
    assert written == nbytes
    torch.cuda.synchronize()
    got = buf.cpu().numpy()
    want = orc.payload_write(fields, [download(dl) for _, dl, _, _ in stack], tokens, logits)
    assert want.size == nbytes
    np.testing.assert_array_equal(got[:nbytes], want)
    assert (got[nbytes:] == 0xAB).all()
    # restore into fresh layers
    fresh = [_fresh_like(shape, dl, wa, wi) for shape, dl, wa, wi in stack]
    tk_h = np.zeros(pos + 10, np.uint32)
    lg_h = np.zeros(vocab, np.float32)
    s, n = abi.ds4c_payload_read(info, cfgs, [f.state for f in fresh], 0, buf.data_ptr(), nbytes, tk_h, lg_h,
                                 stream)
    abi.check(s, "ds4c_payload_read")
    assert n == pos
    np.testing.assert_array_equal(tk_h[:pos], tokens)
    np.testing.assert_array_equal(lg_h, logits)
    # a header written for another runtime shape is refused, and nothing is restored
    other = abi.PayloadInfo(*fields)
    other.vocab_size = vocab + 1
    probe = _fresh_like(*stack[2])
    before = [t.clone() for t in _tensors(probe)]
    s, _ = abi.ds4c_payload_read(other, cfgs, [probe.state] * 8, 0, buf.data_ptr(), nbytes, tk_h,
                                 np.zeros(vocab + 1, np.float32), stream)
    assert s == abi.DS4C_ERR_SHAPE
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(before, _tensors(probe)))
    # resume: the same chunk on the uninterrupted and on the restored stack
    for li, ((shape, dl, _, _), d2) in enumerate(zip(stack, fresh)):
        tk1, o1 = _run_chunk(dl, shape, w.seed, pos, more, li)
        tk2, o2 = _run_chunk(d2, shape, w.seed, pos, more, li)
        dl.sync()
        d2.sync()
        assert torch.equal(o1, o2), f"layer {li} attention"
        if tk1 is not None:
            assert torch.equal(tk1, tk2), f"layer {li} top-k"
        n_live = min(pos + more, shape.swa)
        for a, b in zip(_tensors(dl), _tensors(d2)):
            if a is dl.raw:
                continue
            assert torch.equal(a, b), f"layer {li} state"
        for p in range(pos + more - n_live, pos + more):
            assert torch.equal(dl.raw[0, p % shape.swa], d2.raw[0, p % shape.swa])
