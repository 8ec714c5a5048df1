#!/usr/bin/env python
"""Benchmark of the compressed-KV attention path on one GB300 (or N replicas).

Default workload: one long-context ratio-4 layer, 131072-token prefill in
4096-token chunks (projections, fused compressor, indexer top-k, sparse SWA
attention, ring commit), then the logical-order checkpoint gather.  One step =
that whole pass.  Metric: prefill tokens/s per layer.  The decode step of 32
sequences at 65536 context is measured alongside (``decode`` key).

Prints one JSON line (rank 0).  ``--impl reference`` times the plain-C oracle
on the host cores on a bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from compressed_kv_sparse_compressor_gb300 import configs  # noqa: E402

METRIC = "prefill tokens/s per layer"
# dram__bytes_read.sum + dram__bytes_write.sum of one attention launch (4096 queries), from an ncu capture
# under profiles/; None when the kernel has changed since the counters were taken
ATTN_TRAFFIC = 556817920 + 580525312   # profiles/attn_tc_kernel_prefill_8192tok_chunk2.md
ATTN_TRAFFIC_SRC = "ncu, one 4096-query launch of the 8192-token case (same units per launch as C5)"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--tokens", type=int, default=0, help="override prefill length (profiling only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=256)
    ap.add_argument("--only", default="all", choices=["all", "prefill", "decode"],
                    help="profiling: run only the prefill or only the decode measurement")
    ap.add_argument("--profile-step", action="store_true",
                    help="after timing, run one more step between cudaProfilerStart/Stop (for ncu --profile-from-start off)")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
            "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def attn_flops_chunk(shape, pos0, T):
    """Algorithmic attention flops of one chunk: 4*H*D per (query, row)."""
    rows = 0
    for t in range(pos0, pos0 + T):
        raw = min(t + 1, shape.swa)
        vis = (t + 1) // 4
        rows += raw + min(shape.top_k, vis)
    return 4 * shape.n_heads * shape.head_dim * rows


def indexer_flops_chunk(shape, pos0, T):
    s = sum((t + 1) // 4 for t in range(pos0, pos0 + T))
    return 2 * shape.idx_head_dim * s


class Prefill:
    """C5: the ratio-4 layer prefill + checkpoint gather, inputs resident in HBM."""

    def __init__(self, n_tok: int, device):
        from compressed_kv_sparse_compressor_gb300.layer import DeviceLayer
        w = configs.C5
        self.w = w
        self.shape = shape = w.layer
        self.T = n_tok
        self.chunk = w.chunk
        self.n_chunks = (n_tok + self.chunk - 1) // self.chunk
        self.dl = DeviceLayer(shape, comp_cap=n_tok // 4, idx_cap=n_tok // 4, max_rows=self.chunk)
        wa = configs.lane_weights(shape, w.seed, 0, "attn", device=device)
        wi = configs.lane_weights(shape, w.seed, 0, "idx", device=device)
        self.dl.set_weights(wa, wi)
        D, H, d = shape.head_dim, shape.n_heads, shape.idx_head_dim
        self.h = torch.empty(n_tok, shape.d_model, dtype=torch.bfloat16, device=device)
        self.q = torch.empty(n_tok, H, D, device=device)
        self.q_idx = torch.empty(n_tok, d, device=device)
        self.raw = torch.empty(n_tok, D, device=device)
        for c in range(self.n_chunks):
            p0, n = c * self.chunk, min(self.chunk, n_tok - c * self.chunk)
            self.h[p0:p0 + n] = configs.hidden(shape, w.seed, n, offset_tok=p0, device=device)
            q, qi, r = configs.queries(shape, w.seed, n, offset_tok=p0, device=device)
            self.q[p0:p0 + n], self.q_idx[p0:p0 + n], self.raw[p0:p0 + n] = q, qi, r
        self.out = torch.empty(n_tok, H, D, device=device)
        self.topk = torch.empty(n_tok, shape.top_k, dtype=torch.int32, device=device)
        self.ck = torch.empty(self.dl.checkpoint_floats(n_tok), device=device)
        torch.cuda.synchronize()
        self.events = None

    def inputs(self):
        return [self.h, self.q, self.q_idx, self.raw]

    def outputs(self):
        return [self.out, self.topk, self.ck]

    def step(self, timing=False):
        dl = self.dl
        ev = []
        if timing:
            mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        dl.state_init()
        for c in range(self.n_chunks):
            p0, n = c * self.chunk, min(self.chunk, self.T - c * self.chunk)
            sl = slice(p0, p0 + n)
            if timing:
                e = [mk() for _ in range(5)]
                e[0].record()
                # the projection GEMM and the fused compressor timed apart (event between them)
                dl.compress_prefill_timed(self.h[sl], p0, e[4])
            else:
                dl.compress_prefill(self.h[sl], p0)
            if timing:
                e[1].record()
            dl.indexer_topk(self.q_idx[sl], [p0], 1, n, self.topk[sl])
            if timing:
                e[2].record()
            dl.attention(self.q[sl], self.raw[sl], self.topk[sl], [p0], 1, n, self.out[sl], commit_ring=True)
            if timing:
                e[3].record()
                ev.append(("chunk", p0, n, e))
        if timing:
            g0, g1 = mk(), mk()
            g0.record()
        dl.checkpoint_gather(0, self.T, self.ck)
        if timing:
            g1.record()
            ev.append(("gather", 0, 0, [g0, g1]))
            self.events = ev

    def launches_per_step(self):
        # state init: 5 fills; per chunk: GEMM 1 and its tail reduce 1 (a 4096-row chunk's 320 output
        # tiles leave a partly filled last round on the SMs), fused compressor 1 (both lanes, pool and
        # frontier), score 1, top-k 1, raw mirror 1, attention 1, ring 1; then the gather
        return 5 + 8 * self.n_chunks + 1

    def breakdown(self):
        """Per-call device time (ms) of the last timed step."""
        t = {"compress": 0.0, "indexer_topk": 0.0, "attention": 0.0, "gather": 0.0, "compress_projection": 0.0,
             "compress_fused_pool": 0.0}
        for kind, p0, n, e in self.events:
            if kind == "gather":
                t["gather"] += e[0].elapsed_time(e[1])
            else:
                t["compress"] += e[0].elapsed_time(e[1])
                t["compress_projection"] += e[0].elapsed_time(e[4])
                t["compress_fused_pool"] += e[4].elapsed_time(e[1])
                t["indexer_topk"] += e[1].elapsed_time(e[2])
                t["attention"] += e[2].elapsed_time(e[3])
        return t


def run_ours(args, rank, world, local_rank):
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    from compressed_kv_sparse_compressor_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    if world > 1:
        torch.distributed.barrier()
    if args.only == "decode":
        P, _ = peaks()
        dec = run_decode(device, P, profile=args.profile_step)
        return {"metric": "decode step us at 64K ctx", "value": dec["us_per_step"], "unit": "us", "n_gpus": world,
                "higher_is_better": False, "data": "synthetic", "config": {"workload": dec["workload"]}, "decode": dec}
    n_tok = args.tokens or configs.C5.n_tok
    pf = Prefill(n_tok, device)
    for _ in range(max(args.warmup, 3)):
        pf.step()
    pf.dl.sync()
    clocks = Clocks(local_rank)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    barrier()
    torch.cuda.synchronize()
    clocks.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(args.steps):
        pf.step(timing=(i == args.steps - 1))
    t1.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    pf.dl.sync()
    if args.profile_step:
        torch.cuda.profiler.start()
        pf.step()
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    ms_max, value = aggregate(ms, n_tok, device)
    br = pf.breakdown()

    # roofline of every prefill call (the dominant one is the line's "roofline")
    P, src = peaks()
    shape = pf.shape
    fma = fma_peak_measured(device)
    roofs = {k: roofline(k, br, pf, P, src, fma) for k in ("attention", "indexer_topk", "compress", "compressor")}
    dominant = max(("compress", "indexer_topk", "attention"), key=lambda k: br[k])
    roof = roofs[dominant]

    # checkpoint restore of the step's final state (outside the timed step): scatter the
    # gathered body back into the layer, rebuilding the attention's bf16 mirror
    restore = None
    if args.only != "decode":
        ts = []
        for _ in range(4):
            r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            r0.record()
            pf.dl.checkpoint_scatter(0, pf.T, pf.ck)
            r1.record()
            torch.cuda.synchronize()
            ts.append(r0.elapsed_time(r1))
        pf.dl.sync()
        rms = statistics.median(ts[1:])
        body = pf.ck.numel() * 4
        mirror = (pf.T // 4) * shape.head_dim * (4 + 4)           # comp rows read, bf16 hi / lo written
        rbytes = 2 * body + mirror
        restore = {"ms": round(rms, 4), "bytes": rbytes, "achieved_gbs": round(rbytes / (rms * 1e-3) / 1e9, 1),
                   "hbm_frac": round(rbytes / (rms * 1e-3) / 1e9 / P["hbm_gbs"], 4)}

    # end to end: host (pinned) inputs copied in, results read back, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(pf, args, device)
    dec = None
    if not args.no_decode and args.only == "all":
        dec = run_decode(device, P)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_sample)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_max, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16-in/f32-acc", "data": "synthetic",
        "config": {"workload": configs.C5.name, "layers": 1, "tokens": n_tok, "chunk": pf.chunk,
                   "ratio": 4, "head_dim": shape.head_dim, "idx_head_dim": shape.idx_head_dim,
                   "heads": shape.n_heads, "top_k": shape.top_k, "swa": shape.swa,
                   "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (each 4096-token chunk reads 537 MB of queries)"},
        "gpu_launches": pf.launches_per_step() * args.steps,
        "clocks": clk,
        "roofline": roof,
        "rooflines": roofs,
        "breakdown_ms": {k: round(v, 3) for k, v in br.items()},
        "e2e": e2e,
        "decode": dec,
        "checkpoint_restore": restore,
        "cpu_baseline": cpu,
    }
    return line


def aggregate(ms_local: float, units_per_rank: int, device):
    """Replicas: the step time is the maximum over ranks, the value the units all
    ranks processed per second of that time.  Returns (ms_max, value)."""
    world = torch.distributed.get_world_size() if torch.distributed.is_initialized() else 1
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world * units_per_rank / (ms_max / 1e3)


def fma_peak_measured(device):
    """fp32 FMA rate of this GPU in TFLOP/s, measured in this run with the
    library's register-only fmaf probe (best of 5 launches, CUDA events)."""
    from compressed_kv_sparse_compressor_gb300 import abi
    blocks = torch.cuda.get_device_properties(device).multi_processor_count * 8
    out = torch.empty(blocks * 256, device=device)
    stream = torch.cuda.current_stream(device).cuda_stream
    best = 0.0
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        st, flops = abi.ds4c_fma_probe(blocks, 4096, out.data_ptr(), stream)
        e1.record()
        torch.cuda.synchronize()
        abi.check(st, "ds4c_fma_probe")
        best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    return best


def roofline(kind, br, pf, P, src, fma_peak=None):
    shape, T, C = pf.shape, pf.T, pf.chunk
    n_launch = pf.n_chunks
    if kind == "attention":
        flops = sum(attn_flops_chunk(shape, c * C, min(C, T - c * C)) for c in range(pf.n_chunks))
        per_launch = flops / n_launch
        dur = br["attention"] / n_launch / 1e3
        peak = P["bf16_tflops"]
        return {"kernel": "sparse_swa_attention", "bound": "tensor", "achieved": round(per_launch / dur / 1e12, 2),
                "peak": peak, "unit": "TFLOP/s", "frac": round(per_launch / dur / 1e12 / peak, 4),
                "traffic": ATTN_TRAFFIC, "traffic_source": ATTN_TRAFFIC_SRC, "peak_source": src,
                "units_per_launch": f"{C} queries"}
    if kind == "indexer_topk":
        flops = sum(indexer_flops_chunk(shape, c * C, min(C, T - c * C)) for c in range(pf.n_chunks))
        per_launch = flops / n_launch
        dur = br["indexer_topk"] / n_launch / 1e3
        fsrc = "measured in this run: register-only fp32 fmaf probe (ds4c_fma_probe)"
        if not fma_peak:
            fma_peak = 152 * 128 * 2 * P.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
            fsrc = "152 SMs x 128 fp32 FMA/clk x 2 x max SM clock"
        return {"kernel": "indexer_score_topk", "bound": "alu", "achieved": round(per_launch / dur / 1e12, 2),
                "peak": round(fma_peak, 1), "unit": "TFLOP/s", "frac": round(per_launch / dur / 1e12 / fma_peak, 4),
                "traffic": None, "peak_source": fsrc, "units_per_launch": f"{C} queries",
                "note": "score flops only; the time includes the top-k"}
    if kind == "compressor":
        # the fused compressor kernel alone (store + APE, pool, RMSNorm, tail RoPE, FP8, append, frontier):
        # reads kv and score of both lanes once, writes the appended rows and the attention lane's bf16 mirror
        rd = 4 * (2 * 2 * shape.head_dim + 2 * 2 * shape.idx_head_dim)
        wr = (4 * shape.head_dim + 2 * 2 * shape.head_dim + 4 * shape.idx_head_dim) / 4
        per_launch = (rd + wr) * T / n_launch
        dur = br["compress_fused_pool"] / n_launch / 1e3
        peak = P["hbm_gbs"]
        return {"kernel": "fused_compressor", "bound": "hbm", "achieved": round(per_launch / dur / 1e9, 1),
                "peak": peak, "unit": "GB/s", "frac": round(per_launch / dur / 1e9 / peak, 4), "traffic": None,
                "peak_source": src, "units_per_launch": f"{C} tokens",
                "bytes_per_token": rd + wr,
                "note": "event-timed between the projection GEMM and the next call; the projection output it "
                        "reads was just written by the GEMM and may be served from L2"}
    # compress: projection GEMM flops
    n_out = 2 * 2 * shape.head_dim + 2 * 2 * shape.idx_head_dim
    flops = 2 * T * n_out * shape.d_model
    per_launch = flops / n_launch
    dur = br["compress_projection"] / n_launch / 1e3
    peak = P["bf16_tflops"]
    return {"kernel": "compressor_projection_gemm", "bound": "tensor", "achieved": round(per_launch / dur / 1e12, 2),
            "peak": peak, "unit": "TFLOP/s", "frac": round(per_launch / dur / 1e12 / peak, 4), "traffic": None,
            "peak_source": src, "units_per_launch": f"{C} tokens"}


def run_e2e(pf, args, device):
    """The prefill through the public API from pinned host memory: per chunk, the
    inputs go up on one copy stream, the chunk runs on the compute stream once
    they have landed, and its outputs come back on a second copy stream, so the
    copies of neighbouring chunks overlap the compute (as a serving loop would)."""
    host_in = [t.cpu().pin_memory() for t in pf.inputs()]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in pf.outputs()]
    dev_in, dev_out = pf.inputs(), pf.outputs()
    s_up, s_comp, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    dl = pf.dl
    steps = max(3, min(args.steps, 6))

    def one_step():
        with torch.cuda.stream(s_comp):
            dl.state_init()
        for c in range(pf.n_chunks):
            p0, n = c * pf.chunk, min(pf.chunk, pf.T - c * pf.chunk)
            sl = slice(p0, p0 + n)
            with torch.cuda.stream(s_up):
                for d, h in zip(dev_in, host_in):
                    d[sl].copy_(h[sl], non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s_up)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(landed)
                dl.compress_prefill(pf.h[sl], p0)
                dl.indexer_topk(pf.q_idx[sl], [p0], 1, n, pf.topk[sl])
                dl.attention(pf.q[sl], pf.raw[sl], pf.topk[sl], [p0], 1, n, pf.out[sl], commit_ring=True)
                done = torch.cuda.Event()
                done.record(s_comp)
            with torch.cuda.stream(s_down):
                s_down.wait_event(done)
                host_out[0][sl].copy_(dev_out[0][sl], non_blocking=True)     # out
                host_out[1][sl].copy_(dev_out[1][sl], non_blocking=True)     # topk
        with torch.cuda.stream(s_comp):
            dl.checkpoint_gather(0, pf.T, pf.ck)
            done = torch.cuda.Event()
            done.record(s_comp)
        with torch.cuda.stream(s_down):
            s_down.wait_event(done)
            host_out[2].copy_(dev_out[2], non_blocking=True)                 # checkpoint
        torch.cuda.synchronize()        # a step ends when its last output is on the host

    one_step()                      # warm-up of the streams and the pinned buffers
    torch.cuda.synchronize()
    each = []
    t0 = time.perf_counter()
    for _ in range(steps):
        t1 = time.perf_counter()
        one_step()                  # ends with a device synchronize
        each.append((time.perf_counter() - t1) * 1e3)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    dl.sync()
    bi = sum(t.numel() * t.element_size() for t in host_in)
    bo = sum(t.numel() * t.element_size() for t in host_out)
    # the host link alone: the same bytes copied one way at a time, pinned host memory, one stream
    link = {}
    for name, pairs in (("h2d", list(zip(dev_in, host_in))), ("d2h", list(zip(host_out, dev_out)))):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for dst, src in pairs:
            dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        link[name + "_gbs"] = round((bi if name == "h2d" else bo) / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)
    return {"value": round(pf.T / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": round(ms, 3), "ms_each_step": [round(x, 1) for x in each], "steps": steps,
            "median_step_ms": round(statistics.median(each), 3),
            "host_link": link,
            "host_link_ms": {"h2d": round(bi / (link["h2d_gbs"] * 1e9) * 1e3, 1),
                             "d2h": round(bo / (link["d2h_gbs"] * 1e9) * 1e3, 1)},
            "pipeline": "per chunk: upload, compute and download on three streams; host_link: the step's bytes "
                        "copied one direction at a time on one stream, measured after the timed steps"}


def run_decode(device, P, profile=False):
    """C4: 32 sequences at 65536 + (b mod 4); state built by the compressor, ring from raw rows."""
    from compressed_kv_sparse_compressor_gb300.layer import DeviceLayer
    w = configs.C4
    shape = w.layer
    B = w.n_seq
    lens = [w.ctx + (b % 4) for b in range(B)]
    cap = (max(lens) + 1) // 4 + 1
    dl = DeviceLayer(shape, comp_cap=cap, idx_cap=cap, n_seq=B, max_rows=4096)
    dl.set_weights(configs.lane_weights(shape, w.seed, 0, "attn", device=device),
                   configs.lane_weights(shape, w.seed, 0, "idx", device=device))
    dl.state_init()
    saved = dl.state
    for b in range(B):
        dl.state = dl.seq_view(b)
        for p0 in range(0, lens[b], 4096):
            n = min(4096, lens[b] - p0)
            dl.compress_prefill(configs.hidden(shape, w.seed, n, offset_tok=p0, device=device, layer=b), p0)
        dl.state = saved
        _, _, raw = configs.queries(shape, w.seed, shape.swa, offset_tok=lens[b] - shape.swa, device=device, layer=b)
        for i, p in enumerate(range(lens[b] - shape.swa, lens[b])):
            dl.raw[b, p % shape.swa] = raw[i]
    hid = torch.cat([configs.hidden(shape, w.seed, 1, offset_tok=lens[b], device=device, layer=b) for b in range(B)])
    qs = [configs.queries(shape, w.seed, 1, offset_tok=lens[b], device=device, layer=b) for b in range(B)]
    q = torch.cat([x[0] for x in qs])
    q_idx = torch.cat([x[1] for x in qs])
    raw = torch.cat([x[2] for x in qs])
    topk = torch.empty(B, shape.top_k, dtype=torch.int32, device=device)
    out = torch.empty(B, shape.n_heads, shape.head_dim, device=device)
    snap = [t.clone() for t in (dl.attn_comp, dl.attn_kv, dl.attn_score, dl.idx_comp, dl.idx_kv, dl.idx_score, dl.raw)]
    live = (dl.attn_comp, dl.attn_kv, dl.attn_score, dl.idx_comp, dl.idx_kv, dl.idx_score, dl.raw)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    times = []
    for i in range(23):
        for d_, s_ in zip(live, snap):
            d_.copy_(s_)
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        dl.compress_decode(hid, lens)
        dl.indexer_topk(q_idx, lens, B, 1, topk)
        dl.attention(q, raw, topk, lens, B, 1, out, commit_ring=True)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1) * 1e3)
    dl.sync()
    if profile:
        torch.cuda.profiler.start()
        dl.compress_decode(hid, lens)
        dl.indexer_topk(q_idx, lens, B, 1, topk)
        dl.attention(q, raw, topk, lens, B, 1, out, commit_ring=True)
        torch.cuda.synchronize()
        torch.cuda.profiler.stop()
    us = statistics.median(times)
    # algorithmic bytes: weights + indexer rows scanned + gathered rows + q/out/raw
    wbytes = 2 * (2 * 2 * shape.head_dim + 2 * 2 * shape.idx_head_dim) * shape.d_model
    scan = sum(((L + 1) // 4) * shape.idx_head_dim * 4 for L in lens)
    gath = B * (shape.swa + shape.top_k) * shape.head_dim * 4
    qo = B * (2 * shape.n_heads * shape.head_dim + shape.head_dim + shape.idx_head_dim) * 4
    total = wbytes + scan + gath + qo
    return {"workload": w.name, "us_per_step": round(us, 2), "unit": "us", "higher_is_better": False,
            "algorithmic_bytes": total, "achieved_gbs": round(total / (us * 1e-6) / 1e9, 1),
            "hbm_frac": round(total / (us * 1e-6) / 1e9 / P["hbm_gbs"], 4), "l2": "256 MiB buffer written between steps"}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample(n_tok: int):
    """Time the oracle on n_tok tokens at the end of the C5 layer (positions
    131072 - n_tok ..): compressor, indexer top-k and attention per token, on
    a synthetic steady-state (32768 compressed rows)."""
    import numpy as np
    import oracle as orc
    orc.build()
    w = configs.C5
    shape = w.layer
    T = w.n_tok
    pos0 = T - n_tok
    L = orc.Layer(d_model=shape.d_model, head_dim=shape.head_dim, n_rot=shape.n_rot, idx_head_dim=shape.idx_head_dim,
                  n_heads=shape.n_heads, ratio=4, swa=shape.swa, top_k=shape.top_k, comp_cap=T // 4, idx_cap=T // 4,
                  bf16=True, rms_eps=shape.rms_eps, attn_scale=shape.attn_scale, rope_base=shape.rope_base)
    st = orc.State(L)
    orc.state_init(st)
    rng = np.random.default_rng(0)
    st.attn.comp[:] = rng.standard_normal(st.attn.comp.shape, dtype=np.float32)
    st.idx.comp[:] = rng.standard_normal(st.idx.comp.shape, dtype=np.float32)
    st.raw[:] = rng.standard_normal(st.raw.shape, dtype=np.float32)

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    wa = configs.lane_weights(shape, w.seed, 0, "attn")
    wi = configs.lane_weights(shape, w.seed, 0, "idx")
    wa = (u16(wa[0]), u16(wa[1]), wa[2].numpy(), wa[3].numpy())
    wi = (u16(wi[0]), u16(wi[1]), wi[2].numpy(), wi[3].numpy())
    h = u16(configs.hidden(shape, w.seed, n_tok, offset_tok=pos0))
    q, q_idx, raw = (x.numpy() for x in configs.queries(shape, w.seed, n_tok, offset_tok=pos0))
    t0 = time.perf_counter()
    orc.compress(st, wa, wi, h, pos0)
    tk = orc.indexer_topk(st, q_idx, np.arange(pos0, pos0 + n_tok))
    orc.attention(st, q, raw, tk, pos0)
    orc.ring_commit(st, raw, pos0)
    dt = time.perf_counter() - t0
    return n_tok / dt, orc.num_threads(), dt


def cpu_baseline(n_tok):
    v, cores, dt = oracle_sample(n_tok)
    return {"value": round(v, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_tok} tokens at positions {configs.C5.n_tok - n_tok}..{configs.C5.n_tok - 1} of the "
                      f"131072-token ratio-4 layer (compressor, indexer top-k over 32768 rows, attention over "
                      f"640 rows x 64 heads), {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    n = args.cpu_sample
    for _ in range(args.warmup):
        oracle_sample(max(16, n // 8))
    vals, times = [], []
    for _ in range(args.steps):
        v, cores, dt = oracle_sample(n)
        vals.append(v)
        times.append(dt)
    value = n * len(times) / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": configs.C5.name, "layers": 1, "tokens_per_step_sample": n},
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{n} tokens per step at the end of the 131072-token ratio-4 layer"},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
