#!/usr/bin/env python3
"""Benchmark of the NVFP4 block-scaled linear layer on GB300.

Headline (one JSON line on rank 0): decode W4A16 throughput in HBM GB/s of
the 27B-shaped dense decoder's linears - fused gate/up 5120 -> 34816 and down
17408 -> 5120 at M in {1, 4, 8, 32} tokens. One step runs all eight linears
once; each call streams a different replica of the weights (six replicas,
0.9 GB, so no call finds its weights in the 129 MB L2). Steps are CUDA-graph
replays timed with CUDA events on the launching stream.

Beside the headline the same line carries:
  roofline      the decode GEMV's achieved bytes/s over the measured HBM copy
                bandwidth, and its DRAM traffic from the committed ncu summary
  cpu_baseline  the CPU oracle on a bounded sample of the same workload
  e2e           the same metric through the public API with pinned host
                buffers (host->device inputs, device->host outputs per step)
  clocks        nvidia-smi samples taken while the steps ran
  rows          the other steps of the hot path: W4A4 prefill TFLOPS (of the
                FP4 peak), quantiser GB/s, masked / full draft head GB/s, MoE

--impl reference runs the CPU oracle (the only reference implementation this
path has) on the same metric and workload, on a bounded sample per step.

Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torchrun, one replica per GPU (the path does not shard), max time over ranks.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "NVFP4 GEMM: decode HBM GB/s (% of peak); prefill TFLOPS (% FP4 peak)"
WORKLOAD = ("decode linears of a 27B-shaped dense decoder, NVFP4 W4A16: fused gate/up K=5120->N=34816 and "
            "down K=17408->N=5120 at M in {1,4,8,32} tokens; weights N(0,0.02) quantised per-16 along K, "
            "activations bf16 N(0,1), bf16 out")
DECODE_MATS = (("gate_up", 34816, 5120), ("down", 5120, 17408))
DECODE_M = (1, 4, 8, 32)
REPLICAS = 6
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 : BF16 tensor ratio of GB300
L2_FLUSH_BYTES = 512 << 20


def decode_bytes(N, K, M):
    """Algorithmic bytes of one W4A16 call: packed codes, block scales, the
    bf16 activations read and the bf16 outputs written."""
    return N * K // 2 + N * K // 16 + 2 * M * K + 2 * M * N


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 7:
                    rows.append(parts)
        os.unlink(self.path)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ distributed

def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------- helpers

def gpu_normal(shape, std, seed, dtype=None):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(*shape, generator=g, device="cuda", dtype=torch.float32) * std
    return x if dtype is None else x.to(dtype)


def gpu_student_t(shape, df, seed):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    z = torch.randn(*shape, generator=g, device="cuda")
    chi2 = torch.zeros(*shape, device="cuda")
    for _ in range(df):
        chi2 += torch.randn(*shape, generator=g, device="cuda") ** 2
    return (z / torch.sqrt(chi2 / df)).to(torch.bfloat16)


def capture(fn):
    import torch
    fn()                                   # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


_CLEAN = {}


def l2_flush(flush):
    """Write `flush` (larger than L2), then read a clean buffer of the same
    size: the written lines are evicted (and written back) here, so the timed
    replay that follows starts from an L2 holding only clean, unrelated data
    and pays no write-back of the flush."""
    import torch
    flush.zero_()
    clean = _CLEAN.get(flush.numel())
    if clean is None:
        clean = _CLEAN[flush.numel()] = torch.zeros(flush.numel() // 4, dtype=torch.float32, device=flush.device)
    clean.sum()


def time_graph(g, reps, warmup=5, flush=None):
    """Median ms per replay over `reps` replays, each bracketed by its own CUDA
    events on the launching stream, after `warmup` untimed replays. With
    `flush`, L2 is flushed before every replay and only the replay is timed
    (the flush keeps the GPU busy while the replay is enqueued, so no launch
    gap enters the timing)."""
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        if flush is not None:
            l2_flush(flush)
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def time_graph_mean(g, reps, warmup=5):
    """Mean ms per replay of `reps` back-to-back replays between two events
    (graphs whose replays are chained by programmatic dependent launch, whose
    overlap a per-replay event pair would break)."""
    import torch
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


# sources of the dominant decode kernel; the committed DRAM-traffic record is
# used only while their contents match the hash it was taken with
TRAFFIC_SOURCES = ["nvfp4_block_scaled_04_gb300/csrc/common.cuh", "nvfp4_block_scaled_04_gb300/csrc/tc_util.cuh",
                   "nvfp4_block_scaled_04_gb300/csrc/gemv_core.cuh", "nvfp4_block_scaled_04_gb300/csrc/gemv_tma.cuh",
                   "nvfp4_block_scaled_04_gb300/csrc/gemv.cu"]


def traffic_hash():
    import hashlib
    h = hashlib.sha256()
    for s in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(kernel_key, src_files):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel sources changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            data = json.load(f)
        entry = data[kernel_key]
        h = hashlib.sha256()
        for s in src_files:
            with open(os.path.join(ROOT, s), "rb") as f:
                h.update(f.read())
        if entry.get("source_sha256") != h.hexdigest()[:16]:
            return None
        return entry["dram_bytes_per_launch"]
    except Exception:
        return None


# ----------------------------------------------------------- decode setup

class Decode:
    """Weights (six replicas per matrix), activations, outputs, workspaces."""

    def __init__(self, nv):
        import torch
        self.nv = nv
        self.w = {}
        for i, (name, N, K) in enumerate(DECODE_MATS):
            wf = gpu_normal((N, K), 0.02, seed=100 + i)
            q = nv.quantize(wf)
            del wf
            self.w[name] = [q] + [nv.QTensor(q.codes.clone(), q.scales.clone(), q.s_t.clone(), N, K)
                                  for _ in range(REPLICAS - 1)]
        self.x, self.y, self.ws = {}, {}, {}
        for M in DECODE_M:
            for name, N, K in DECODE_MATS:
                self.x[(M, name)] = gpu_normal((M, K), 1.0, seed=200 + M, dtype=torch.bfloat16)
                self.y[(M, name)] = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
                self.ws[(M, name)] = torch.empty(nv.workspace_size(nv.OP_GEMM_W4A16, M, N, K), dtype=torch.uint8,
                                                 device="cuda")
        torch.cuda.synchronize()

    def calls(self):
        return [(M, name, N, K) for M in DECODE_M for name, N, K in DECODE_MATS]

    def call(self, M, name, rep):
        self.nv.gemm_w4a16(self.x[(M, name)], self.w[name][rep], out=self.y[(M, name)],
                           workspace=self.ws[(M, name)])

    def step_fn(self, step_index):
        calls = self.calls()

        def fn():
            for j, (M, name, _, _) in enumerate(calls):
                self.call(M, name, (len(calls) * step_index + j) % REPLICAS)
        return fn

    def step_bytes(self):
        return sum(decode_bytes(N, K, M) for M, _, N, K in self.calls())


def e2e_graph(dec):
    """One step through the public API with pinned host buffers: every call's
    activations are copied host -> device and its output device -> host.
    The copies run on a second stream, as a serving loop would issue them: all
    uploads at the start of the step, each output read back as soon as its
    call has finished, while the next calls compute."""
    import torch
    hx = {k: v.cpu().pin_memory() for k, v in dec.x.items()}
    hy = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in dec.y.items()}
    calls = dec.calls()
    copies = torch.cuda.Stream()

    def fn():
        main = torch.cuda.current_stream()
        copies.wait_stream(main)
        uploaded = []
        with torch.cuda.stream(copies):
            for M, name, _, _ in calls:
                dec.x[(M, name)].copy_(hx[(M, name)], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(copies)
                uploaded.append(ev)
        for j, (M, name, _, _) in enumerate(calls):
            main.wait_event(uploaded[j])
            dec.call(M, name, j % REPLICAS)
            done = torch.cuda.Event()
            done.record(main)
            copies.wait_event(done)
            with torch.cuda.stream(copies):
                hy[(M, name)].copy_(dec.y[(M, name)], non_blocking=True)
        main.wait_stream(copies)
    h2d = sum(v.numel() * v.element_size() for v in hx.values())
    d2h = sum(v.numel() * v.element_size() for v in hy.values())
    return capture(fn), h2d, d2h


def measure_silu_mul(nv, peaks, reps):
    """The 27B gate/up with SiLU * mul fused (h [M][17408] written once)
    against the plain gate/up GEMV (y [M][34816] written, then read back by a
    separate SiLU * mul): per call, weights rotated over six replicas."""
    import torch
    N, K = 34816, 5120
    wf = gpu_normal((N, K), 0.02, seed=100)
    q = nv.quantize(wf)
    del wf
    reps_w = [q] + [nv.QTensor(q.codes.clone(), q.scales.clone(), q.s_t.clone(), N, K) for _ in range(REPLICAS - 1)]
    res = {}
    for M in DECODE_M:
        x = gpu_normal((M, K), 1.0, seed=300 + M, dtype=torch.bfloat16)
        h = torch.empty(M, N // 2, dtype=torch.bfloat16, device="cuda")
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(nv.workspace_size(nv.OP_GEMM_W4A16, M, N, K), dtype=torch.uint8, device="cuda")
        gf = capture(lambda: [nv.gemm_w4a16_silu_mul(x, reps_w[r % REPLICAS], out=h, workspace=ws)
                              for r in range(12)])
        gp = capture(lambda: [nv.gemm_w4a16(x, reps_w[r % REPLICAS], out=y, workspace=ws) for r in range(12)])
        tf, tp = time_graph(gf, 20) / 12, time_graph(gp, 20) / 12
        b = decode_bytes(N, K, M) - 2 * M * N + 2 * M * (N // 2)
        res[f"M{M}"] = {"us_fused": tf * 1e3, "us_plain_gemv": tp * 1e3, "gbs_fused": b / tf / 1e6,
                        "frac_hbm_fused": b / tf / 1e6 / peaks["hbm_gbs"],
                        "bytes_saved_vs_unfused": 4 * M * N}
    return res


# --------------------------------------------------------- the other rows

def measure_rows(nv, peaks, reps):
    import torch
    out = {}
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16

    # the FP4 tensor pipe's own ceiling: one CTA per SM issuing block-scaled
    # 128 x 256 x 64 MMAs from shared memory, no global traffic
    n_mma = 20000
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    gp = capture(lambda: nv.probe_fp4_mma_rate(n_mma))
    clk = ClockSampler(torch.cuda.current_device()).start()
    tp = time_graph(gp, reps)
    ck = clk.stop()
    probe_tflops = sms * n_mma * 2.0 * 128 * 256 * 64 / tp / 1e9
    out["fp4_ceiling_measured"] = {"tflops": probe_tflops, "ms": tp, "ctas": sms, "mma_per_cta": n_mma,
                                   "instruction": "tcgen05.mma.cta_group::1.kind::mxf4nvf4 128x256x64",
                                   "sm_mhz_median": ck["sm_mhz"], "clock_reasons": ck["reasons"]}
    del gp

    # prefill W4A4, M=8192 K=5120 N=34816
    M, K, N = 8192, 5120, 34816
    a = gpu_student_t((M, K), 4, seed=3)
    wf = gpu_normal((N, K), 0.02, seed=4)
    qw = nv.prepack_scales(nv.quantize(wf))
    del wf
    qa = nv.quantize(a, scale_layout=nv.SCALES_MMA)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g = capture(lambda: nv.gemm_w4a4(qa, qw, out=y))
    t = time_graph(g, reps)
    qws = torch.empty(nv.workspace_size(nv.OP_QUANTIZE, M, 0, K), dtype=torch.uint8, device="cuda")

    def q_and_gemm():
        q = nv.quantize(a, scale_layout=nv.SCALES_MMA, workspace=qws)
        nv.gemm_w4a4(q, qw, out=y)
    g2 = capture(q_and_gemm)
    t2 = time_graph(g2, reps)
    gq = capture(lambda: nv.quantize(a, scale_layout=nv.SCALES_MMA, workspace=qws))
    tq = time_graph(gq, reps, flush=flush)
    flops = 2.0 * M * N * K
    out["w4a4_prefill"] = {
        "shape": [M, N, K], "ms": t, "tflops": flops / t / 1e9, "frac_fp4_peak": flops / t / 1e9 / fp4_peak,
        "fp4_peak_tflops": fp4_peak, "peak_basis": f"{peaks['source']} bf16 x {FP4_OVER_BF16:g}",
        "frac_fp4_ceiling_measured": flops / t / 1e9 / probe_tflops,
        "ms_with_quantize": t2, "tflops_with_quantize": flops / t2 / 1e9}
    qbytes = M * K * 2 + M * K // 2 + M * K // 16
    out["quantize_activations"] = {"shape": [M, K], "ms": tq, "gbs": qbytes / tq / 1e6,
                                   "frac_hbm": qbytes / tq / 1e6 / peaks["hbm_gbs"]}

    # the same GEMM handing its output on as NVFP4 (the next W4A4 layer's
    # input): fused epilogue with a given tensor scale, the dynamic two-pass
    # form, and the unfused bf16 GEMM + quantiser it replaces
    st_out = torch.tensor([0.05], device="cuda")
    wsq = torch.empty(nv.workspace_size(nv.OP_GEMM_W4A4_QUANT, M, N, K), dtype=torch.uint8, device="cuda")
    codes_o = torch.empty(M, N // 2, dtype=torch.uint8, device="cuda")
    gf = capture(lambda: nv.gemm_w4a4_quant(qa, qw, s_t=st_out, workspace=wsq))
    tf = time_graph(gf, reps)
    gd = capture(lambda: nv.gemm_w4a4_quant(qa, qw, y=y, workspace=wsq))
    td = time_graph(gd, reps)
    qws2 = torch.empty(nv.workspace_size(nv.OP_QUANTIZE, M, 0, N), dtype=torch.uint8, device="cuda")
    gu = capture(lambda: (nv.gemm_w4a4(qa, qw, out=y), nv.quantize(y, scale_layout=nv.SCALES_MMA, workspace=qws2)))
    tu = time_graph(gu, reps)
    out["w4a4_to_nvfp4"] = {
        "shape": [M, N, K], "ms_fused_given_scale": tf, "ms_dynamic_scale_two_pass": td, "ms_unfused": tu,
        "tflops_fused": flops / tf / 1e9, "bf16_round_trip_bytes_saved_fused": 2 * M * N * 2,
        "note": "unfused = bf16 GEMM output written, then read twice by the quantiser (amax + encode)"}
    del a, qa, qw, y, g, g2, gq, gf, gd, gu, codes_o
    torch.cuda.empty_cache()

    # masked draft head: 248,320 x 5120, 32,768-id mask, M in {1, 4, 8}
    V, K = 248320, 5120
    wf = gpu_normal((V, K), 0.02, seed=5)
    qh = nv.quantize(wf)
    del wf
    gperm = torch.Generator(device="cuda")
    gperm.manual_seed(6)
    # one 32,768-id mask per draft step, so no step finds its rows still in L2
    # (six: the steady-state chains below rotate over all of them, 566 MB)
    masks = [torch.randperm(V, generator=gperm, device="cuda")[:32768].to(torch.int32) for _ in range(6)]
    qmasks = [nv.gather_rows(qh, ix) for ix in masks]   # one-time prepack: masked rows as compact matrices
    head = {}
    for Mh in (1, 4, 8):
        hs = [gpu_normal((Mh, K), 1.0, seed=7 + s, dtype=torch.bfloat16) for s in range(3)]
        wss = [torch.zeros(nv.workspace_size(nv.OP_GATHER_ARGMAX, Mh, V, K), dtype=torch.uint8, device="cuda")
               for _ in range(3)]

        def steps(kind):
            def fn():   # the page's three draft steps
                for s in range(3):
                    if kind == "masked":
                        nv.gemv_argmax(hs[s], qmasks[s], masks[s], workspace=wss[s])
                    elif kind == "gathered":
                        nv.gather_gemv_argmax(hs[s], qh, masks[s], workspace=wss[s])
                    else:
                        nv.gather_gemv_argmax(hs[s], qh, None, workspace=wss[s])
            return fn
        res = {}
        for label, kind, rows in (("masked", "masked", 32768), ("masked_gathered_in_place", "gathered", 32768),
                                  ("full", "full", V)):
            g = capture(steps(kind))
            t = time_graph(g, reps, flush=flush) / 3
            b = rows * (K // 2 + K // 16) + 2 * Mh * K
            res[label] = {"ms": t, "gbs": b / t / 1e6, "frac_hbm": b / t / 1e6 / peaks["hbm_gbs"]}
        res["full_over_masked_time"] = res["full"]["ms"] / res["masked"]["ms"]
        # steady state: draft steps chained back to back (12 per graph, the six
        # compact masks in turn, 566 MB, so no step finds its rows in L2), as a
        # serving loop runs them between verifications
        hs6 = [gpu_normal((Mh, K), 1.0, seed=20 + s, dtype=torch.bfloat16) for s in range(6)]
        ws6 = [torch.zeros(nv.workspace_size(nv.OP_GATHER_ARGMAX, Mh, V, K), dtype=torch.uint8, device="cuda")
               for _ in range(6)]
        gs = capture(lambda: [nv.gemv_argmax(hs6[s % 6], qmasks[s % 6], masks[s % 6], workspace=ws6[s % 6])
                              for s in range(12)])
        t = time_graph(gs, reps) / 12
        b = 32768 * (K // 2 + K // 16) + 2 * Mh * K
        res["masked_steady_state"] = {"ms": t, "gbs": b / t / 1e6, "frac_hbm": b / t / 1e6 / peaks["hbm_gbs"]}
        del gs
        head[f"M{Mh}"] = res
    head["bytes_ratio_full_over_masked"] = V / 32768
    head["timing"] = ("per draft step: graphs of 3 steps (one mask and hidden state each), L2 flushed per graph; "
                      "masked_steady_state: graphs of 12 chained steps over six masks")
    out["draft_head"] = head

    # speculative verify: 8 sequences x (3 drafts + 1) = 32 rows against the
    # full vocabulary, greedy acceptance fused into the argmax's last CTA
    B, D = 8, 3
    hv = [gpu_normal((B * (D + 1), K), 1.0, seed=40 + s, dtype=torch.bfloat16) for s in range(3)]
    drafts = torch.randint(0, V, (B, D), generator=gperm, device="cuda", dtype=torch.int64).to(torch.int32)
    wsv = torch.zeros(nv.workspace_size(nv.OP_GATHER_ARGMAX, B * (D + 1), V, K), dtype=torch.uint8, device="cuda")
    g = capture(lambda: [nv.verify_accept(hv[s], qh, drafts, workspace=wsv) for s in range(3)])
    t = time_graph(g, reps, flush=flush) / 3
    b = V * (K // 2 + K // 16) + 2 * B * (D + 1) * K
    out["verify_head"] = {"rows": B * (D + 1), "ms": t, "gbs": b / t / 1e6, "frac_hbm": b / t / 1e6 / peaks["hbm_gbs"],
                          "timing": "per verify step: graphs of 3 steps, L2 flushed per graph"}
    del qh, qmasks
    torch.cuda.empty_cache()

    # MoE: 128 experts, top-8, H=2048, I=768
    E, H, I, k = 128, 2048, 768, 8
    w13 = nv.quantize_stack([gpu_normal((2 * I, H), 0.02, seed=1000 + e) for e in range(E)])
    w2 = nv.quantize_stack([gpu_normal((H, I), 0.02, seed=2000 + e) for e in range(E)])
    w13m, w2m = nv.prepack_scales(w13), nv.prepack_scales(w2)   # MMA-layout scales for the W4A4 layer
    moe, moe4 = {}, {}
    wbytes = E * (2 * I * H + H * I) * (1 / 2 + 1 / 16)
    for T in (256, 4096):
        logits = gpu_normal((T, E), 1.0, seed=8)
        x = gpu_normal((T, H), 1.0, seed=9, dtype=torch.bfloat16)
        o = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(nv.workspace_size(nv.OP_GROUPED_GEMM, T, H, I, E, k), dtype=torch.uint8, device="cuda")

        def layer():
            ids, wts = nv.moe_route(logits, k)
            nv.grouped_gemm(x, ids, wts, w13, w2, out=o, workspace=ws)
        g = capture(layer)
        t = time_graph(g, reps, flush=flush)
        flops = 2.0 * T * k * (2 * I * H + H * I)
        b = wbytes + 4 * T * H
        moe[f"T{T}"] = {"ms": t, "gbs": b / t / 1e6, "frac_hbm": b / t / 1e6 / peaks["hbm_gbs"],
                        "tflops": flops / t / 1e9, "frac_bf16_peak": flops / t / 1e9 / peaks["bf16_tflops"]}
        ws4 = torch.empty(nv.workspace_size(nv.OP_GROUPED_GEMM_W4A4, T, H, I, E, k), dtype=torch.uint8, device="cuda")

        def layer4():
            ids, wts = nv.moe_route(logits, k)
            nv.grouped_gemm_w4a4(x, ids, wts, w13m, w2m, out=o, workspace=ws4)
        g4 = capture(layer4)
        t4 = time_graph(g4, reps, flush=flush)
        moe4[f"T{T}"] = {"ms": t4, "gbs": b / t4 / 1e6, "frac_hbm": b / t4 / 1e6 / peaks["hbm_gbs"],
                         "tflops": flops / t4 / 1e9, "frac_fp4_ceiling_measured": flops / t4 / 1e9 / probe_tflops}
        del g4, ws4
    out["moe"] = moe
    out["moe_w4a4"] = moe4
    return out


# ------------------------------------------------------------- CPU oracle
#
# The oracle (numpy) runs in child processes started with OMP_NUM_THREADS,
# OPENBLAS_NUM_THREADS and MKL_NUM_THREADS set to 1, so each child computes on
# exactly one core: one child alone gives the single-core figure, one child
# per available host core (each on its own sample of weight rows, all at
# once) the all-core figure. The decode weights are drawn once by the parent
# and shared with the children through memory-mapped .npy files.

PIN_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def host_cores():
    """(os.cpu_count(), cores this process may run on = nproc)."""
    n_all = os.cpu_count() or 1
    try:
        n_aff = len(os.sched_getaffinity(0))
    except Exception:
        n_aff = n_all
    return n_all, n_aff


def prepare_oracle_weights(tmpdir):
    """The decode weights on the host (CPU generator) as .npy files, and the
    oracle's tensor scale of each (fp32, exact as a Python float)."""
    import numpy as np

    import oracle as O
    import synth
    meta = {}
    for name, _, _ in DECODE_MATS:
        w = synth.decode_weight(name).numpy()
        path = os.path.join(tmpdir, f"{name}.npy")
        np.save(path, w)
        meta[name] = {"path": path, "s_t": float(O.tensor_scale(w))}
    return meta


def cpu_leg(args):
    """Child process: the oracle's W4A16 decode on a sample of weight rows per
    call of the eight decode calls (rows quantised by the oracle with the full
    tensor's scale, times the step's activations in fp64). --cpu-rows 0 sizes
    the sample from a 16-row trial so one step takes ~--cpu-budget s. Prints
    {bytes, seconds, rows, step_seconds} for the timed steps."""
    import numpy as np

    import oracle as O
    import synth
    meta = json.loads(args.cpu_meta)
    mats = {name: (np.load(m["path"], mmap_mode="r"), np.float32(m["s_t"])) for name, m in meta.items()}
    xs = {(M, K): synth.decode_activation(M, K).float().numpy() for M in DECODE_M for _, _, K in DECODE_MATS}
    rng = np.random.default_rng(1000 + args.cpu_shard)

    def step(rows):
        b, t = 0, 0.0
        for M in DECODE_M:
            for name, N, K in DECODE_MATS:
                w, st = mats[name]
                r = np.sort(rng.choice(N, min(rows, N), replace=False))
                wr = np.ascontiguousarray(w[r])       # rows read from the shared file: not the oracle's work
                t0 = time.perf_counter()
                q = O.quantize(wr, s_t=st)
                O.gemm_w4a16(xs[(M, K)], q)
                t += time.perf_counter() - t0
                b += len(r) * (K // 2 + K // 16) + 2 * M * K + 2 * M * len(r)
        return b, t

    rows = args.cpu_rows
    if rows <= 0:
        _, t16 = step(16)
        rows = int(max(1, min(4096, 16 * args.cpu_budget / max(t16, 1e-3))))
    for _ in range(args.cpu_warmup):
        step(rows)
    tb, tt, per = 0, 0.0, []
    for _ in range(args.cpu_steps):
        b, t = step(rows)
        tb, tt = tb + b, tt + t
        per.append(t)
    print(json.dumps({"bytes": tb, "seconds": tt, "rows": rows, "step_seconds": per}), flush=True)


def cpu_children(meta, n, rows, steps, warmup, budget=0.0):
    """Run n pinned oracle children at once (shards 0..n-1); their results."""
    env = dict(os.environ, **PIN_ENV)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-leg", "--cpu-meta", json.dumps(meta),
           "--cpu-rows", str(rows), "--cpu-steps", str(steps), "--cpu-warmup", str(warmup), "--cpu-budget",
           str(budget)]
    procs = [subprocess.Popen(cmd + ["--cpu-shard", str(i)], stdout=subprocess.PIPE, env=env, text=True)
             for i in range(n)]
    outs = []
    for p in procs:
        o, _ = p.communicate(timeout=1200)
        if p.returncode != 0:
            raise RuntimeError(f"oracle child exited with {p.returncode}")
        outs.append(json.loads(o.strip().splitlines()[-1]))
    return outs


def cpu_baseline(budget):
    """The oracle on the host: one pinned core, then every available core."""
    n_all, n_aff = host_cores()
    with tempfile.TemporaryDirectory() as d:
        meta = prepare_oracle_weights(d)
        one = cpu_children(meta, 1, 0, 1, 0, budget)[0]
        many = cpu_children(meta, n_aff, one["rows"], 1, 0)
    v1 = one["bytes"] / one["seconds"] / 1e9
    vall = sum(o["bytes"] for o in many) / max(o["seconds"] for o in many) / 1e9
    return {"value": vall, "unit": "GB/s", "cores": n_aff, "kind": "oracle",
            "sample": f"{one['rows']} weight rows per call of the 8 decode calls per process, oracle-quantised and "
                      f"multiplied in fp64; {n_aff} single-threaded processes at once, each its own row sample "
                      f"({max(o['seconds'] for o in many):.1f} s)",
            "host_cores": n_all, "nproc": n_aff, "threads_per_process": 1, "pinning": PIN_ENV,
            "single_core": {"value": v1, "unit": "GB/s", "cores": 1, "seconds": one["seconds"]}}


# ------------------------------------------------------------------ main

def config_block(n):
    return {"workload": WORKLOAD, "l2": f"inputs larger than L2: {REPLICAS} weight replicas (0.9 GB) rotated "
            "so consecutive calls stream different copies", "timing": "CUDA-graph replays, CUDA events on the "
            "launching stream", "replicas": "one independent replica per GPU (the path does not shard)",
            "n_gpus": n}


def run_ours(args):
    import torch
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    import nvfp4_block_scaled_04_gb300 as nv
    nv.lib()
    peaks = load_peaks()
    dec = Decode(nv)
    graphs = [capture(dec.step_fn(i)) for i in range(3)]
    step_bytes = dec.step_bytes()

    # warm-up: W steps, then a ~1 s load window so the clocks settle
    clocks = ClockSampler(local).start()
    for i in range(args.warmup):
        graphs[i % 3].replay()
    torch.cuda.synchronize()
    t_end = time.time() + 1.0
    while time.time() < t_end:
        for i in range(30):
            graphs[i % 3].replay()
        torch.cuda.synchronize()

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(args.steps):
        graphs[i % 3].replay()
    b.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = max_over_ranks(dist, a.elapsed_time(b) / args.steps, f"cuda:{local}")
    clk = clocks.stop()
    value = world * step_bytes / (ms * 1e-3) / 1e9

    # per-call durations of the dominant kernel (graph of 12 calls over the replicas)
    per_call = {}
    tot_b, tot_t = 0.0, 0.0
    for M, name, N, K in dec.calls():
        g = capture(lambda M=M, name=name: [dec.call(M, name, r % REPLICAS) for r in range(12)])
        t = time_graph(g, 20) / 12
        bts = decode_bytes(N, K, M)
        per_call[f"{name}_M{M}"] = {"us": t * 1e3, "gbs": bts / t / 1e6, "frac": bts / t / 1e6 / peaks["hbm_gbs"]}
        tot_b += bts
        tot_t += t
    achieved = tot_b / tot_t / 1e6

    # end to end through the public API with host buffers
    ge, h2d, d2h = e2e_graph(dec)
    te = time_graph(ge, max(10, args.steps // 10))
    e2e = {"value": world * step_bytes / (te * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": te}

    rows = measure_rows(nv, peaks, reps=args.row_reps) if not args.no_rows else {}
    if not args.no_rows:
        rows["gate_up_silu_mul_fused"] = measure_silu_mul(nv, peaks, args.row_reps)

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16xf16->f32 (e2m1/e4m3 weights dequantised exactly to f16)",
            "data": "synthetic (seeded device RNG, distributions of the served layers)",
            "config": config_block(world), "frac_hbm_peak": value / world / peaks["hbm_gbs"],
            "gpu_launches": 16 * args.steps,
            "roofline": {"kernel": "nvfp4_gemm_w4a16 (activation prep + skinny_tma_kernel)", "bound": "hbm",
                         "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"] + " HBM copy",
                         "traffic": read_traffic("skinny_tma_kernel_decode", TRAFFIC_SOURCES),
                         "per_call": per_call},
            "e2e": e2e, "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"],
                                   "reasons": clk["reasons"], "samples": clk["samples"]},
            "rows": rows}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_reference(args):
    """The oracle on the same metric and workload, on every available host
    core (one pinned single-threaded process per core, each its own row
    sample of every step), each step a bounded sample sized so the whole run
    stays within a few minutes. Rank 0 only."""
    world, rank, _ = dist_info()
    if rank != 0:
        return
    n_all, n_aff = host_cores()
    budget = min(8.0, 100.0 / max(1, args.steps + args.warmup))
    with tempfile.TemporaryDirectory() as d:
        meta = prepare_oracle_weights(d)
        rows = cpu_children(meta, 1, 0, 1, 0, budget)[0]["rows"]
        outs = cpu_children(meta, n_aff, rows, args.steps, args.warmup)
    tot_b = sum(o["bytes"] for o in outs)
    wall = max(o["seconds"] for o in outs)
    value = tot_b / wall / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded CPU RNG, distributions of the served layers)", "config": config_block(world),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": n_aff, "kind": "oracle",
                             "sample": f"{rows} weight rows per call of the 8 decode calls per step and process, "
                                       f"{n_aff} single-threaded processes at once",
                             "host_cores": n_all, "nproc": n_aff, "pinning": PIN_ENV},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_case(args):
    """One kernel family at a chosen size, a few launches after warm-up: the
    workload the ncu captures in profiles/ are taken on."""
    import torch
    import nvfp4_block_scaled_04_gb300 as nv
    nv.lib()
    res = {"case": args.case}
    if args.case == "w4a4":
        M, N, K = args.m, 34816, 5120
        a = gpu_student_t((M, K), 4, seed=3)
        qa = nv.quantize(a, scale_layout=nv.SCALES_MMA)
        qw = nv.prepack_scales(nv.quantize(gpu_normal((N, K), 0.02, seed=4)))
        y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        g = capture(lambda: nv.gemm_w4a4(qa, qw, out=y))
        t = time_graph(g, 3)
        res.update(shape=[M, N, K], ms=t, tflops=2.0 * M * N * K / t / 1e9)
    elif args.case == "quantize":
        M, K = args.m, 5120
        a = gpu_student_t((M, K), 4, seed=3)
        ws = torch.empty(nv.workspace_size(nv.OP_QUANTIZE, M, 0, K), dtype=torch.uint8, device="cuda")
        g = capture(lambda: nv.quantize(a, scale_layout=nv.SCALES_MMA, workspace=ws))
        res.update(shape=[M, K], ms=time_graph(g, 3))
    elif args.case == "draft":
        V, K = 248320, 5120
        qh = nv.quantize(gpu_normal((V, K), 0.02, seed=5))
        gp = torch.Generator(device="cuda")
        gp.manual_seed(6)
        idx = torch.randperm(V, generator=gp, device="cuda")[:32768].to(torch.int32)
        h = gpu_normal((args.m, K), 1.0, seed=7, dtype=torch.bfloat16)
        g = capture(lambda: nv.gather_gemv_argmax(h, qh, idx))
        res.update(M=args.m, ms=time_graph(g, 3))
    elif args.case in ("moe", "moe_w4a4"):
        E, H, I = 128, 2048, 768
        w13 = nv.quantize_stack([gpu_normal((2 * I, H), 0.02, seed=1000 + e) for e in range(E)])
        w2 = nv.quantize_stack([gpu_normal((H, I), 0.02, seed=2000 + e) for e in range(E)])
        if args.case == "moe_w4a4":
            w13, w2 = nv.prepack_scales(w13), nv.prepack_scales(w2)
        logits = gpu_normal((args.m, E), 1.0, seed=8)
        x = gpu_normal((args.m, H), 1.0, seed=9, dtype=torch.bfloat16)
        fn = nv.grouped_gemm_w4a4 if args.case == "moe_w4a4" else nv.grouped_gemm

        def layer():
            ids, wts = nv.moe_route(logits, 8)
            fn(x, ids, wts, w13, w2)
        g = capture(layer)
        res.update(T=args.m, ms=time_graph(g, 3))
    torch.cuda.synchronize()
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--row-reps", type=int, default=50, help="timed replays per row (median)")
    ap.add_argument("--no-rows", action="store_true", help="skip the non-headline rows")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work per core for cpu_baseline")
    ap.add_argument("--case", choices=["w4a4", "quantize", "draft", "moe", "moe_w4a4"], default=None,
                    help="run one kernel family only (the profiling workloads)")
    ap.add_argument("--m", type=int, default=2048, help="rows / tokens for --case")
    # the oracle child processes of the CPU legs
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-meta", default="{}", help=argparse.SUPPRESS)
    ap.add_argument("--cpu-rows", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-steps", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-warmup", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--cpu-shard", type=int, default=0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_leg:
        cpu_leg(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
