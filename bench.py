#!/usr/bin/env python
"""Benchmark of the DSpark hot path on one GB300: one step = one decode cycle
(draft -> schedule -> pack -> verify) over a batch of synthetic inputs.

Metric: committed tokens per second (accepted drafts + one bonus token per
request) over the device time of draft + schedule + pack + verify; the
target-model stand-in (a row gather of precomputed synthetic target logits
into the packed buffer) sits between pack and verify and is not timed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) each rank runs an independent replica on its own GPU
(the path shards by request; there is no data-path collective) and rank 0
prints the aggregate.  --impl reference times the CPU oracle on a bounded
sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/s (draft+schedule+verify) at vocab 152K; % HBM roofline"
UNIT = "tokens/s"
# what `value` counts (the metric's tokens): every accepted draft plus the one
# bonus (or replacement) token each request commits per cycle
VALUE_COUNTS = ("committed tokens per second: accepted drafts + one bonus token per request, over the device "
                "time of draft + schedule + pack + verify; verified target rows per second are given beside it")
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e nominal, for the fraction the pages' ~8 TB/s figure asks for
FLUSH_BYTES = 256 << 20
OTHER_WORKLOADS = ("tiny_chain", "rejection_sampling", "pctree", "mixed_traffic")


def status_bits(status):
    """Names of the device status bits set (the informational tier bit included)."""
    from speculative_decoding_markov_gb300 import binding as sdm
    names = {sdm.DEV_BAD_TOKEN: "bad_token", sdm.DEV_TIER_UNCAPTURED: "tier_uncaptured (informational)",
             sdm.DEV_TIMEOUT: "timeout", sdm.DEV_BAD_WINDOW: "bad_window", sdm.DEV_CAPACITY: "capacity",
             sdm.DEV_BAD_CLASS: "bad_class", sdm.DEV_TIER_OVERFLOW: "tier_overflow"}
    return [n for b, n in names.items() if status & b]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--no-graphs", action="store_true", help="launch eagerly instead of replaying CUDA graphs")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_chain")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the oracle sample")
    ap.add_argument("--no-workloads", action="store_true",
                    help="only the selected workload (by default a run of the headline workload also times the "
                         "other four workloads, shorter, and reports them under `workloads`)")
    ap.add_argument("--workload-steps", type=int, default=200, help="timed cycles of each of the other workloads")
    ap.add_argument("--scheduler", default="budget", choices=["budget", "dynamic", "threshold"],
                    help="threshold: the conventional fixed confidence threshold (--tau); "
                         "budget: the early-stopping scheduler on the additive table; dynamic: the production "
                         "scheduler (capacity from the confidences of two steps before, global search over the "
                         "tier-stepped table)")
    ap.add_argument("--tau", type=float, default=0.5, help="confidence threshold of --scheduler threshold")
    ap.add_argument("--head", default="markov", choices=["markov", "rnn"],
                    help="sequential head of the chain draft: the Markov head, or the RNN head (memo recurrence; "
                         "dense tensor-core projection per step)")
    ap.add_argument("--requests", type=int, default=0,
                    help="run the workload with this many requests instead (smaller cases for profiler captures)")
    ap.add_argument("--observe", action="store_true",
                    help="add the fused observability pass to every verify: the soft label 1 - TV(q, p) of every "
                         "verified row and the cycle statistics (ceiling histograms per class, per-position accept "
                         "counts, calibration bins and ECE)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s sustained, source): the measured copy
    bandwidth and GEMM throughput of this GPU, else the fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops_sustained", d.get("bf16_tflops", 1700.0))), "measured"
    return 6800.0, 1700.0, "fallback"


def measured_burst_tflops(default):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f).get("bf16_tflops", default))
    return 1900.0


KERNEL_SOURCES = {   # the files whose text fixes each reported kernel's code
    "chain_scan_kernel+chain_pick_kernel": ("chain_pruned.cu", "schedule_pack.cuh", "device.cuh", "internal.h"),
    "markov_gemm_kernel<sample>+draft_select_kernel": ("markov_gemm.cu", "select.cu", "device.cuh", "internal.h"),
    "markov_gemm_kernel<tree>+tree_select_kernel": ("markov_gemm.cu", "select.cu", "device.cuh", "internal.h"),
    "markov_gemm_kernel<tree_lse>+tree_level_kernel": ("markov_gemm.cu", "tree_pruned.cu", "tree_common.cuh",
                                                       "chain_pruned.cu", "schedule_pack.cuh", "device.cuh",
                                                       "internal.h"),
    "row_stream_kernel<argmax>": ("stream.cu", "device.cuh", "internal.h"),
}


def kernel_source_hash(kernel: str = "chain_scan_kernel+chain_pick_kernel"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_markov_gb300", "csrc")
    for f in KERNEL_SOURCES.get(kernel, ()):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed ncu summary profiles/traffic.txt (one line per kernel
    and workload: name, workload, source hash, bytes), if it was taken on the
    current kernel sources; None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
                return int(parts[3]) if parts[2] == kernel_source_hash(kernel) else None
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)                    # let the sampler start before the work
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self, t0=None, t1=None):
        """Median SM clock and active throttle reasons of the samples taken
        between wall-clock times t0 and t1 (all samples if fewer than 3 fall
        inside)."""
        import datetime
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        rows = []
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:8]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside, window = rows, "warm-up and timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
class Cycle:
    """Preallocated buffers and the launch sequence of one decode cycle."""

    def __init__(self, w, seed, device, dynamic=False, observe=False, tau=None, rnn=False):
        import torch

        from speculative_decoding_markov_gb300 import binding as sdm
        from speculative_decoding_markov_gb300 import synthetic

        self.torch, self.sdm, self.synthetic = torch, sdm, synthetic
        self.w = w
        self.dev = device
        self.inp = synthetic.generate(w, seed=seed, device=device)
        R, B, V, r = w.R, w.B, w.V, w.r
        self.sample = w.decode == "sample"
        self.tree = w.decode == "tree"
        self.dynamic = dynamic
        self.tau = tau
        self.rnn = rnn and not self.tree
        self.obs = observe and not self.tree
        i32 = dict(dtype=torch.int32, device=device)
        self.status = sdm.new_status(device)
        self.side = torch.cuda.Stream(device=device)
        self.layout_ready = torch.cuda.Event()
        self.prepared = None
        if self.tree:
            self._init_tree(R, B, V, r, i32)
            return
        self.mode = {"compact": sdm.COMPACT, "static": sdm.STATIC, "cap_accept": sdm.CAP_ACCEPT}[w.modes[0]]
        self.dr = dict(tokens=torch.empty((R, B), **i32), logq=torch.zeros((R, B), dtype=torch.float32, device=device),
                       lse=torch.zeros((R, B), dtype=torch.float32, device=device))
        self.sc = dict(survival=torch.empty((R, B), dtype=torch.float32, device=device), budget=torch.empty((R,), **i32),
                       expected=torch.empty((1,), dtype=torch.float64, device=device),
                       total_tokens=torch.empty((1,), **i32), capacity=torch.empty((1,), **i32))
        cap = sdm.pack_capacity(R, B, list(w.tiers))
        self.cap = cap
        self.pk = dict(cu_seqlens=torch.empty((R + 1,), **i32), packed_tok=torch.empty((cap,), **i32),
                       packed_req=torch.empty((cap,), **i32), packed_pos=torch.empty((cap,), **i32),
                       tier=torch.empty((1,), **i32))
        tdt = synthetic.torch_dtype(w.target_dtype)
        self.packed = torch.empty((cap, V), dtype=tdt, device=device)
        self.vr = dict(accept=torch.empty((R,), **i32), ceiling=torch.empty((R,), **i32),
                       out_tok=torch.empty((R, B + 1), **i32), n_out=torch.empty((R,), **i32))
        self.ws_draft = sdm.workspace(sdm.OP_DRAFT_CHAIN_RNN if self.rnn else sdm.OP_DRAFT_CHAIN, R, B, V, r,
                                      device=device)
        if self.rnn:
            self.inp.update(synthetic.rnn_inputs(w, seed=seed, device=device))
        self.ws_verify = sdm.workspace(sdm.OP_VERIFY, R, B, V, r, cap, device=device)
        if self.obs:
            self.n_class, self.n_bins = len(w.sigma), 10
            self.cls = synthetic.request_class(w, seed).to(torch.int32).to(device)
            self.label = torch.empty((R, B), dtype=torch.float32, device=device)
            self.ws_label = sdm.workspace(sdm.OP_TV_LABEL, R, B, V, r, cap, device=device)
            nc, nb = self.n_class, self.n_bins
            self.st = dict(hist=torch.empty((nc, B + 1), **i32), reached=torch.empty((nc, B), **i32),
                           hits=torch.empty((nc, B), **i32), bin_n=torch.empty((nb,), **i32),
                           bin_hit=torch.empty((nb,), **i32),
                           bin_conf=torch.empty((nb,), dtype=torch.float64, device=device),
                           ece=torch.empty((1,), dtype=torch.float64, device=device))
            self.side2 = torch.cuda.Stream(device=device)
        # greedy drafting uses the Markov head's prepared tables, built once
        # per weights (model-load time, outside the timed cycle)
        self.prepared = None if (self.sample or self.rnn) else sdm.markov_prepare(self.inp["U"], self.inp["W"])
        # one untimed cycle fixes the drafted prefix; the stand-in target model
        # then provides every window row along it
        self.draft()
        self.schedule_pack()
        self.target = synthetic.chain_target(self.inp, self.dr["tokens"], w.target_dtype)
        self.gather()
        self.verify()
        torch.cuda.synchronize()
        assert int(self.status.item()) & ~sdm.DEV_TIER_UNCAPTURED == 0, f"device status {int(self.status.item())}"

    def _init_tree(self, R, B, V, r, i32):
        """PCTree cycle: tree draft (batched frontier, per-level prune, global
        top-N) and greedy verification of every tree slot."""
        torch, sdm, w = self.torch, self.sdm, self.w
        S = w.N + 1
        dev = self.dev
        self.tr = dict(tok=torch.empty((R, S), **i32), parent=torch.empty((R, S), **i32),
                       depth=torch.empty((R, S), **i32), score=torch.empty((R, S), dtype=torch.float32, device=dev),
                       mask=torch.empty((R, S, (S + 31) // 32), **i32), n_nodes=torch.empty((R,), **i32))
        self.vr = dict(accept=torch.empty((R,), **i32), out_tok=torch.empty((R, B + 1), **i32),
                       n_out=torch.empty((R,), **i32))
        self.ws_draft = sdm.workspace(sdm.OP_DRAFT_TREE, R, B, V, r, w.P, w.k, w.N, device=dev)
        self.ws_verify = sdm.workspace(sdm.OP_VERIFY_TREE, R, B, V, 0, 0, 0, w.N, device=dev)
        # the level by bound pruning needs the Markov head's prepared tables,
        # built once per weights (model-load time, outside the timed cycle)
        self.prepared = sdm.markov_prepare(self.inp["U"], self.inp["W"])
        self.draft()
        self.target = self.synthetic.tree_target(self.inp, self.tr["tok"], self.tr["depth"], self.tr["n_nodes"],
                                                 w.target_dtype)
        self.verify()
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0, f"device status {int(self.status.item())}"

    def verified_rows(self):
        if self.tree:
            return int(self.tr["n_nodes"].sum().item())
        return int(self.pk["cu_seqlens"][-1].item())

    # the four timed operations -------------------------------------------
    def draft(self):
        sdm, i = self.sdm, self.inp
        if self.tree:
            w = self.w
            sdm.draft_tree(i["L"], i["U"], i["W"], i["anchor"], w.k, w.P, w.N, out=self.tr, ws=self.ws_draft,
                           dev_status=self.status, prepared=self.prepared)
            return
        if self.rnn:
            sdm.draft_chain_rnn(i["L"], i["U"], i["W"], i["A_rnn"], i["X_rnn"], i["anchor"],
                                decode=sdm.SAMPLE if self.sample else sdm.GREEDY, temperature=self.w.temperature,
                                seed=0, cycle=0, out=self.dr, ws=self.ws_draft, dev_status=self.status)
            return
        sdm.draft_chain(i["L"], i["U"], i["W"], i["anchor"], decode=sdm.SAMPLE if self.sample else sdm.GREEDY,
                        temperature=self.w.temperature, seed=0, cycle=0, out=self.dr, ws=self.ws_draft,
                        dev_status=self.status, prepared=self.prepared)

    def schedule(self):
        sdm, i = self.sdm, self.inp
        if self.tau is not None:
            sdm.schedule_threshold(i["conf"], self.tau, out=self.sc, dev_status=self.status)
        elif self.dynamic:
            sdm.schedule_dynamic(i["conf"], i["conf_stale"], i["cost_tiered"], out=self.sc, dev_status=self.status)
        else:
            sdm.schedule_budget(i["conf"], i["cost"], out=self.sc, dev_status=self.status)

    def pack(self):
        sdm, i = self.sdm, self.inp
        budget = self.sc["budget"] if self.mode == sdm.COMPACT else None
        sdm.pack_ragged(i["anchor"], self.dr["tokens"], budget, i["tiers"], out=self.pk, dev_status=self.status)

    def schedule_pack(self):
        if self.tree:    # the tree's node budget is its global top-N
            return
        self.schedule()
        self.pack()

    def front(self):
        """Draft, schedule and pack.  The budget needs only the confidences.
        With the greedy chain's prepared tables and a scan that fills the GPU,
        the scheduler and the ragged layout run in one extra CTA of the draft's
        scan and the pick writes its tokens into the layout (one call).
        Otherwise the scheduler runs on a side stream while the draft runs;
        with the prepared tables the side stream also lays out the windows and
        the pick fills them (no pack pass after the draft), else the pack
        joins both."""
        if self.tree:
            self.draft()
            return
        torch, sdm, i = self.torch, self.sdm, self.inp
        main = torch.cuda.current_stream()
        self.side.wait_stream(main)
        fused = self.prepared is not None and not self.rnn
        if fused and self.front_one_launch():
            # the scheduler and the layout in the draft's own first launch
            # (one extra CTA of the scan), the pick filling the layout
            sdm.draft_chain_front(i["L"], i["U"], i["W"], i["anchor"], self.prepared, i["conf"], i["cost"],
                                  i["tiers"], use_budget=self.mode == sdm.COMPACT, tokens=self.dr["tokens"],
                                  sched=self.sc, pk=self.pk, ws=self.ws_draft, dev_status=self.status)
            return
        with torch.cuda.stream(self.side):
            self.schedule()
            if fused:
                budget = self.sc["budget"] if self.mode == sdm.COMPACT else None
                sdm.pack_ragged(i["anchor"], None, budget, i["tiers"], out=self.pk, dev_status=self.status,
                                gamma=self.w.B)
                self.layout_ready.record(self.side)
        if fused:
            sdm.draft_chain_packed(i["L"], i["U"], i["W"], i["anchor"], self.prepared, self.pk["cu_seqlens"],
                                   self.pk["packed_tok"], tokens=self.dr["tokens"], layout_ready=self.layout_ready,
                                   ws=self.ws_draft, dev_status=self.status)
            main.wait_stream(self.side)
            return
        self.draft()
        main.wait_stream(self.side)
        self.pack()

    def gather(self):
        if self.tree:    # the target rows of every tree slot are resident
            return
        self.synthetic.gather_packed(self.target, self.pk["packed_req"], self.pk["packed_pos"], out=self.packed)

    def verify(self):
        sdm, i = self.sdm, self.inp
        if self.tree:
            sdm.verify_tree(self.target, self.tr["tok"], self.tr["parent"], self.tr["n_nodes"], self.w.B, out=self.vr,
                            ws=self.ws_verify, dev_status=self.status)
            return
        kw = {}
        if self.sample:
            kw = dict(logq=self.dr["logq"], lse_q=self.dr["lse"], L=i["L"], U=i["U"], W=i["W"])
        if self.obs:   # the soft labels need no verify output: they run beside it
            main = self.torch.cuda.current_stream()
            self.side2.wait_stream(main)
            with self.torch.cuda.stream(self.side2):
                self.tv_label()
        sdm.verify(self.mode, sdm.SAMPLE if self.sample else sdm.GREEDY, self.packed, self.pk["cu_seqlens"],
                   i["anchor"], self.dr["tokens"], budget=self.sc["budget"], temperature=self.w.temperature,
                   out=self.vr, ws=self.ws_verify, dev_status=self.status, **kw)
        if self.obs:
            self.stats()
            main.wait_stream(self.side2)

    def tv_label(self):
        i = self.inp
        self.sdm.tv_label(self.packed, self.pk["cu_seqlens"], i["anchor"], self.dr["tokens"], i["L"], i["U"], i["W"],
                          lse_q=self.dr["lse"] if self.sample else None, temperature=self.w.temperature,
                          out=self.label, ws=self.ws_label, dev_status=self.status)

    def stats(self):
        self.sdm.observe(self.inp["conf"], self.pk["cu_seqlens"], self.vr["ceiling"], self.cls, self.n_class,
                         self.n_bins, out=self.st, dev_status=self.status)

    def front_one_launch(self):
        """Whether the budget scheduler and the layout ride in the draft's scan
        (sdm_draft_chain_front): the budget scheduler, its shared memory within
        the 48 KB the scan is launched with, and a scan that fills every SM
        (four 32 KB items per SM or more).  Only then does a side-stream
        scheduler wait for the scan to drain; on a smaller scan it runs beside
        it at once, with four times the threads of the scan's extra CTA."""
        if self.tau is not None or self.dynamic or self.prepared is None or self.rnn or self.tree:
            return False
        esz = 4 if self.w.l_dtype == self.sdm.FP32 else 2
        items = self.w.R * self.w.B * -(-self.w.V * esz // (32 * 1024))
        if items < 4 * self.torch.cuda.get_device_properties(0).multi_processor_count:
            return False
        n = self.w.R * self.w.B
        n_pad = 1
        while n_pad < n:
            n_pad <<= 1
        smem = n_pad * 8 + 256 * 8 + self.w.R * 4 + n * 4 + (n_pad + 1) * 4
        return n <= 8192 and smem <= 48 * 1024

    def launches_per_step(self):
        if self.tree:   # init, scan, per level the GEMM and the level kernel, finalize; verify stream and walk
            return (2 * self.w.B + 3) + 2
        if self.rnn:   # per step the memo update and the GEMM (+ the select when sampling); greedy: fill, finalize
            draft = self.w.B * (3 if self.sample else 2) + (0 if self.sample else 2)
        else:
            draft = 2 if self.prepared is not None else self.w.B + 2
        verify = 5 if self.sample else 2
        if self.obs:   # row stream, row list, [draft log-sum-exp pass + reduction], label pass + reduction, stats
            verify += 5 if self.sample else 7
        schedule_pack = 0 if self.front_one_launch() else 2   # inside the draft's scan, or two launches
        return draft + schedule_pack + verify

    def capture(self):
        """CUDA graphs of the two timed segments (the stand-in gather between
        them stays outside)."""
        torch = self.torch
        self.g_draft = torch.cuda.CUDAGraph()
        self.g_verify = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_draft):
            self.front()
        with torch.cuda.graph(self.g_verify):
            self.verify()
        torch.cuda.synchronize()


def run_ours(args, w, world, rank, local):
    import torch

    torch.cuda.set_device(local)
    if not hasattr(args, "cpu_threads_seconds"):
        args.cpu_threads_seconds = args.cpu_seconds
    dev = torch.device("cuda", local)
    dynamic = args.scheduler == "dynamic"
    tau = args.tau if args.scheduler == "threshold" else None
    cyc = Cycle(w, seed=rank, device=dev, dynamic=dynamic, observe=args.observe, tau=tau, rnn=args.head == "rnn")
    R, B, V = w.R, w.B, w.V
    committed = int(cyc.vr["n_out"].sum().item())
    accepted = int(cyc.vr["accept"].sum().item())
    windows = cyc.verified_rows()                            # target rows verified per cycle
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    graphs = not args.no_graphs
    if graphs:
        cyc.capture()

    def run_draft():
        if graphs:
            cyc.g_draft.replay()
        else:
            cyc.front()

    def run_verify():
        if graphs:
            cyc.g_verify.replay()
        else:
            cyc.verify()

    def step(ev=None):
        flush.fill_(1)                                      # L2 flush, untimed
        if ev:
            ev[0].record(stream)
        run_draft()                                         # draft + schedule + pack
        if ev:
            ev[1].record(stream)
        cyc.gather()                                        # target stand-in, untimed
        if ev:
            ev[2].record(stream)
        run_verify()
        if ev:
            ev[3].record(stream)

    # draft-only events on a separate eager run give the draft / schedule split
    ev_split = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for _ in range(args.warmup):
        step()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        w0 = time.time()
        for k in range(args.steps):
            step(events[k])
        torch.cuda.synchronize()
        w1 = time.time()
    barrier(world)
    # one eager cycle split into draft and schedule+pack (reported only)
    flush.fill_(1)
    ev_split[0].record(stream)
    cyc.draft()
    ev_split[1].record(stream)
    cyc.schedule_pack()
    ev_split[2].record(stream)
    torch.cuda.synchronize()
    split_draft = ev_split[0].elapsed_time(ev_split[1])
    split_sched = ev_split[1].elapsed_time(ev_split[2])
    t_front = sum(e[0].elapsed_time(e[1]) for e in events) / 1e3       # draft + schedule + pack
    t_verify = sum(e[2].elapsed_time(e[3]) for e in events) / 1e3
    t_total = t_front + t_verify
    # the draft alone (for the roofline of its kernels): its own graph, the
    # same L2 flush before every launch, CUDA events on the stream
    n_draft = max(20, min(200, args.steps))
    g_only = None
    if graphs:
        g_only = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_only):
            cyc.draft()
    ev_d = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_draft)]
    for k in range(n_draft + 3):
        flush.fill_(1)
        if k >= 3:
            ev_d[k - 3][0].record(stream)
        g_only.replay() if g_only is not None else cyc.draft()
        if k >= 3:
            ev_d[k - 3][1].record(stream)
    torch.cuda.synchronize()
    t_draft = sum(e[0].elapsed_time(e[1]) for e in ev_d) / 1e3 / n_draft * args.steps   # seconds per args.steps
    t_max, units = merge_ranks(t_total, [committed * args.steps, windows * args.steps], world)
    status = int(cyc.status.item())
    observe = observe_alone(cyc, flush, stream, graphs, max(20, min(200, args.steps))) if cyc.obs else None

    # roofline of the dominant kernel (algorithmic bytes or flops / measured time)
    hbm_peak, tc_peak, peak_kind = measured_peaks()
    s_l = 2 if w.l_dtype == 0 else 4
    s_t = 2 if w.target_dtype == 0 else 4
    verify_bytes = windows * V * s_t                            # every verified target row once
    if cyc.tree:
        # a level: 2 (R P) r V tensor-core flops (the tree draft is bound by
        # them: 318.6 GFLOP a cycle at R = 32, P = 8, B = 16, r = 256); the
        # bytes a level moves (W, and the level's L rows twice: the scan and
        # the GEMM) reported beside them
        draft_alg, draft_launches, bound = 2.0 * R * w.P * w.r * V, B, "tensor"
        dname = "markov_gemm_kernel<tree_lse>+tree_level_kernel"
    elif cyc.prepared is not None:
        # the greedy chain's algorithmic bytes: every element of L once and W
        # once per cycle; the bound-pruned design itself streams L alone (the
        # few W^T rows it scores come from L2), reported beside it
        draft_alg, draft_launches, bound = float(R * B * V * s_l + w.r * V * 2), 1, "hbm"
        dname = "chain_scan_kernel+chain_pick_kernel"
    else:
        # one GEMM (+ one inverse-CDF select) per step: that step's rows of L
        # and all of W (the RNN head's memo update reads A and U rows only)
        draft_alg, draft_launches, bound = float(R * V * s_l + w.r * V * 2), B, "hbm"
        dname = ("rnn_step_kernel+" if cyc.rnn else "") + (
            "markov_gemm_kernel<sample>+draft_select_kernel" if cyc.sample else "markov_gemm_kernel<greedy>")
    if t_draft >= t_verify:
        kname = dname
        per_launch_s = t_draft / args.steps / draft_launches
        achieved = draft_alg / per_launch_s / (1e12 if bound == "tensor" else 1e9)
    else:
        # the verify path: every verified target row once; sampling adds the
        # residual pass (its L and target rows and W); the soft-label pass,
        # when on, its own bytes
        kname, bound = ("row_stream_kernel<lse>+residual" if cyc.sample else "row_stream_kernel<argmax>"), "hbm"
        if cyc.sample:
            verify_bytes += R * V * (s_l + s_t) + w.r * V * 2
        if observe is not None:
            kname += "+tv_label"
            verify_bytes += observe["algorithmic_bytes"]
        per_launch_s = t_verify / args.steps
        achieved = verify_bytes / per_launch_s / 1e9
    if bound == "tensor":   # a short launch timed alone: the burst rate
        tc_peak = measured_burst_tflops(tc_peak)
    peak, unit = (tc_peak, "TFLOP/s") if bound == "tensor" else (hbm_peak, "GB/s")
    traffic = recorded_traffic(kname, w.name)
    draft_bytes = R * B * V * s_l
    extra = {}
    if kname == dname and cyc.prepared is not None and not cyc.tree:
        extra["achieved_l_only"] = draft_bytes / per_launch_s / 1e9
        extra["frac_l_only"] = extra["achieved_l_only"] / hbm_peak
    if kname == dname and cyc.tree:
        level_bytes = w.r * V * 2 + 2 * R * V * s_l
        extra["hbm_bytes_per_level"] = level_bytes
        extra["hbm_achieved_gbs"] = level_bytes / per_launch_s / 1e9
        extra["hbm_frac"] = extra["hbm_achieved_gbs"] / hbm_peak

    e2e = None
    if not args.no_e2e:
        def make_twin():
            t = Cycle(w, seed=rank, device=dev, dynamic=dynamic, observe=args.observe, tau=tau, rnn=args.head == "rnn")
            if graphs:
                t.capture()
            return t

        e2e = run_e2e(cyc, args, committed, make_twin)

    cpu = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu = oracle_sample(w, cyc.inp, args.cpu_seconds, dynamic, cyc.obs, tau)
        cpu["all_cores"] = oracle_sample_threads(w, cyc.inp, args.cpu_threads_seconds, dynamic, cyc.obs, tau)

    clk = clocks.summary(w0, w1)
    out = {
        "metric": METRIC,
        "value": units[0] / t_max,
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_max / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "R": R, "B": B, "V": V, "r": w.r, "decode": w.decode, "mode": w.modes[0],
                   "scheduler": None if cyc.tree else args.scheduler, "tau": tau, "observe": cyc.obs,
                   "head": None if cyc.tree else args.head,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "l2": "flushed by a 256 MB write before every step",
                   "timed": "draft+schedule+pack+verify (CUDA events); target stand-in row gather excluded"},
        "breakdown_ms_per_step": {"draft+schedule+pack": t_front / args.steps * 1e3,
                                  "verify": t_verify / args.steps * 1e3,
                                  "draft_alone": t_draft / args.steps * 1e3,
                                  "eager_split_ms": {"draft": split_draft, "schedule+pack": split_sched}},
        "graphs": graphs,
        "tokens_per_step": {"committed": committed, "accepted_drafts": accepted, "verified_rows": windows},
        "verified_rows_per_s": units[1] / t_max,
        "value_counts": VALUE_COUNTS,
        "roofline": {"bound": bound, "kernel": kname, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS if bound == "hbm" else None,
                     "nominal_peak": NOMINAL_HBM_GBS if bound == "hbm" else None, "traffic": traffic,
                     "traffic_unit": "DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     **extra,
                     "algorithmic": {"draft_per_launch": draft_alg, "draft_launches_per_cycle": draft_launches,
                                     "draft_unit": "flop" if bound == "tensor" else "byte",
                                     "verify_bytes_per_cycle": verify_bytes, "L_bytes_per_cycle": draft_bytes}},
        "gpu_launches": cyc.launches_per_step() * args.steps,
        "device_status": status,
        "device_status_bits": status_bits(status),
        "clocks": clk,
    }
    if e2e is not None:
        out["e2e"] = e2e
    if observe is not None:
        observe["roofline_frac"] = observe["achieved_gbs"] / hbm_peak
        out["observe"] = observe
    if cpu is not None:
        out["cpu_baseline"] = cpu
    return out


def observe_alone(cyc, flush, stream, graphs, n):
    """The soft-label pass on its own (graph replays after an L2 flush, CUDA
    events on the stream) and what the last cycle's statistics say."""
    import torch

    w = cyc.w
    g = None
    if graphs:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cyc.tv_label()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for k in range(n + 3):
        flush.fill_(1)
        if k >= 3:
            ev[k - 3][0].record(stream)
        g.replay() if g is not None else cyc.tv_label()
        if k >= 3:
            ev[k - 3][1].record(stream)
    torch.cuda.synchronize()
    t = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3 / n
    rows = int((cyc.label >= 0).sum().item())
    s_l = 2 if w.l_dtype == 0 else 4
    s_t = 2 if w.target_dtype == 0 else 4
    passes = 1 if cyc.sample else 2                # the greedy draft returns no log-sum-exp
    # per listed row: its target row twice (log-sum-exp stream, label pass),
    # its L row once per GEMM pass; W once per GEMM pass
    alg = rows * w.V * (2 * s_t + passes * s_l) + passes * w.r * w.V * 2
    lab = cyc.label[cyc.label >= 0]
    return {"label_ms": t * 1e3, "label_rows": rows, "algorithmic_bytes": alg, "achieved_gbs": alg / t / 1e9,
            "mean_label": float(lab.mean().item()) if rows else None, "ece": float(cyc.st["ece"].item()),
            "ceiling_hist": cyc.st["hist"].tolist(), "timed_in_verify": True}


def run_e2e(cyc, args, committed, make_twin):
    """Same cycle through the C-ABI with host buffers: every step copies its
    inputs (backbone logits, anchors, confidences, target logits) from pinned
    host memory and reads the committed tokens back.  Two cycles alternate, as
    a serving loop would: while one computes step k, a copy stream fills the
    other's inputs for step k + 1, so the host link (about 210 GB/s, the
    bound here) and the kernels overlap."""
    import torch

    keys = ("L", "anchor", "conf") + (("conf_stale",) if cyc.dynamic else ()) + (("X_rnn",) if cyc.rnn else ())
    host = {k: cyc.inp[k].cpu().pin_memory() for k in keys}
    host["target"] = cyc.target.cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    # alternate two buffer sets only where the copies are what a step waits
    # for (a few MB and up); a small step gains nothing from the overlap
    pipelined = h2d >= (8 << 20)
    cycles = [cyc, make_twin()] if pipelined else [cyc]
    outs = [(torch.empty_like(c.vr["out_tok"], device="cpu").pin_memory(),
             torch.empty_like(c.vr["n_out"], device="cpu").pin_memory()) for c in cycles]
    d2h = outs[0][0].numel() * 4 + outs[0][1].numel() * 4
    comp = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in cycles]
    done = [torch.cuda.Event() for _ in cycles]

    def copy_inputs(j):
        c = cycles[j]
        if not pipelined:   # on the compute stream, in order
            for k in keys:
                c.inp[k].copy_(host[k], non_blocking=True)
            c.target.copy_(host["target"], non_blocking=True)
            return
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[j])          # its previous step has read them
            for k in keys:
                c.inp[k].copy_(host[k], non_blocking=True)
            c.target.copy_(host["target"], non_blocking=True)
            copied[j].record(copy_stream)

    def compute(j):
        c = cycles[j]
        if pipelined:
            comp.wait_event(copied[j])
        if hasattr(c, "g_draft"):
            c.g_draft.replay()
        else:
            c.front()
        c.gather()
        if hasattr(c, "g_verify"):
            c.g_verify.replay()
        else:
            c.verify()
        outs[j][0].copy_(c.vr["out_tok"], non_blocking=True)
        outs[j][1].copy_(c.vr["n_out"], non_blocking=True)
        if pipelined:
            done[j].record(comp)

    def run(n):
        if not pipelined:   # copy, compute, read back, one step at a time
            for _ in range(n):
                copy_inputs(0)
                compute(0)
                comp.synchronize()
            return
        copy_inputs(0)
        for s in range(n):
            if s + 1 < n:
                copy_inputs((s + 1) % 2)
            compute(s % 2)
        torch.cuda.synchronize()

    run(4)
    k = max(4, min(50, args.steps // 4))
    t0 = time.perf_counter()
    run(k)
    dt = time.perf_counter() - t0
    assert all(int(o[1].sum()) == committed for o in outs)
    return {"value": committed * k / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt / k * 1e3,
            "pipelined": "copies of step k + 1 overlap the kernels of step k" if pipelined else False}


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------
def _np_of(t):
    import numpy as np
    import torch

    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def oracle_front(w, inp, idx, cycle_seed=0, dynamic=False, tau=None):
    """The oracle's draft, schedule (over all requests) and pack for the
    requests idx (the RNN head drafts when inp holds its weights).  Returns
    the state the verify needs."""
    import numpy as np
    import torch

    import oracle

    idx_t = torch.as_tensor(idx, dtype=torch.long, device=inp["L"].device)
    sub = {k: inp[k].index_select(0, idx_t) for k in ("L", "L_bonus", "eta", "anchor")}
    sub["U"], sub["W"] = inp["U"], inp["W"]
    L = _np_of(sub["L"])
    U, W = (inp["_U_np"], inp["_W_np"]) if "_U_np" in inp else (_np_of(inp["U"]), _np_of(inp["W"]))
    an = _np_of(sub["anchor"])
    st = dict(idx=list(idx), sub=sub, L=L, U=U, W=W, an=an, seed=cycle_seed)
    if w.decode == "tree":
        st["tr"] = oracle.draft_tree(L, U, W, an, w.k, w.P, w.N)
        return st
    conf, cost, tiers = _np_of(inp["conf"]), _np_of(inp["cost"]), _np_of(inp["tiers"])
    if dynamic:
        stale, cost = _np_of(inp["conf_stale"]), _np_of(inp["cost_tiered"])
    sample = w.decode == "sample"
    ids = np.asarray(idx, np.int32)
    if "A_rnn" in inp:
        X = _np_of(inp["X_rnn"].index_select(0, idx_t.to(inp["X_rnn"].device)))
        dr = oracle.draft_chain_rnn(L, U, W, _np_of(inp["A_rnn"]), X, an,
                                    decode=oracle.SAMPLE if sample else oracle.GREEDY, temperature=w.temperature,
                                    seed=cycle_seed, req_ids=ids)
    else:
        dr = oracle.draft_chain(L, U, W, an, decode=oracle.SAMPLE if sample else oracle.GREEDY,
                                temperature=w.temperature, seed=cycle_seed, req_ids=ids)
    if tau is not None:
        sc = oracle.schedule_threshold(conf, tau)
    elif dynamic:
        sc = oracle.schedule_dynamic(conf, stale, cost)
    else:
        sc = oracle.schedule_budget(conf, cost)
    budget = sc["budget"][ids]
    static = w.modes[0] != "compact"
    st.update(dr=dr, budget=budget, ids=ids, conf=conf,
              pk=oracle.pack_ragged(an, dr["tokens"], None if static else budget, tiers))
    return st


def oracle_target(w, st):
    """The target stand-in's rows for the oracle's drafts (input synthesis:
    never timed)."""
    import torch

    from speculative_decoding_markov_gb300 import synthetic

    sub = {k: v.cpu() for k, v in st["sub"].items()}
    if w.decode == "tree":
        tr = st["tr"]
        st["target"] = _np_of(synthetic.tree_target(sub, torch.as_tensor(tr["tok"]), torch.as_tensor(tr["depth"]),
                                                    torch.as_tensor(tr["n_nodes"]), w.target_dtype))
        return
    pk = st["pk"]
    tgt = synthetic.chain_target(sub, torch.as_tensor(st["dr"]["tokens"]), w.target_dtype)
    st["target"] = _np_of(synthetic.gather_packed(tgt, torch.as_tensor(pk["packed_req"]),
                                                  torch.as_tensor(pk["packed_pos"])))


def oracle_back(w, st, observe=False):
    """The oracle's verify (and the observability pass) for the state of
    oracle_front; returns the committed tokens."""
    import numpy as np

    import oracle
    from speculative_decoding_markov_gb300 import synthetic

    if w.decode == "tree":
        tr = st["tr"]
        return int(oracle.verify_tree(st["target"], tr["tok"], tr["parent"], tr["n_nodes"], w.B)["n_out"].sum())
    sample = w.decode == "sample"
    dr, pk, an, L, U, W = st["dr"], st["pk"], st["an"], st["L"], st["U"], st["W"]
    mode = {"compact": oracle.COMPACT, "static": oracle.STATIC, "cap_accept": oracle.CAP_ACCEPT}[w.modes[0]]
    kw = {}
    if sample:
        kw = dict(logq=dr["logq"], lse_q=dr["lse"], L=L, U=U, W=W, temperature=w.temperature, seed=st["seed"])
    vr = oracle.verify(mode, oracle.SAMPLE if sample else oracle.GREEDY, st["target"], pk["cu_seqlens"], an,
                       dr["tokens"], budget=st["budget"], req_ids=st["ids"], **kw)
    if observe:
        oracle.tv_label(st["target"], pk["cu_seqlens"], an, dr["tokens"], L, U, W, temperature=w.temperature)
        cls = synthetic.request_class(w, 0).numpy().astype(np.int32)[st["ids"]]
        oracle.observe(st["conf"][st["ids"]], pk["cu_seqlens"], vr["ceiling"], cls, len(w.sigma), 10)
    return int(vr["n_out"].sum())


def oracle_cycle(w, inp, idx, cycle_seed=0, dynamic=False, observe=False, tau=None):
    """One oracle cycle for the requests idx (schedule over all requests);
    returns (seconds of oracle work, committed tokens).  The target stand-in
    between draft and verify is not timed."""
    t0 = time.perf_counter()
    st = oracle_front(w, inp, idx, cycle_seed, dynamic, tau)
    t1 = time.perf_counter()
    oracle_target(w, st)
    t2 = time.perf_counter()
    toks = oracle_back(w, st, observe)
    t3 = time.perf_counter()
    return (t1 - t0) + (t3 - t2), toks


def host_inputs(inp):
    """The workload's inputs in host memory, with the Markov tables as numpy
    arrays once (not per oracle call)."""
    h = {k: v.cpu() for k, v in inp.items()}
    h["_U_np"], h["_W_np"] = _np_of(h["U"]), _np_of(h["W"])
    return h


def oracle_sample(w, inp, seconds, dynamic=False, observe=False, tau=None):
    """Oracle throughput on a bounded sample: requests are added one at a time
    (each a full cycle: its draft, the schedule over all requests, its pack and
    verify) until about `seconds` of oracle work."""
    inp = host_inputs(inp)
    spent, toks, n = 0.0, 0, 0
    while n < w.R and (spent < seconds or n < 2):
        dt, c = oracle_cycle(w, inp, [n], dynamic=dynamic, observe=observe, tau=tau)
        spent += dt
        toks += c
        n += 1
    return {"value": toks / spent, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} of {w.R} requests of one cycle (one cycle each; schedule over all {w.R}), "
                      f"{spent:.1f} s of single-threaded oracle work"}


def host_cores():
    return max(1, len(os.sched_getaffinity(0)))


def oracle_sample_threads(w, inp, seconds, dynamic=False, observe=False, tau=None, threads=None):
    """The same per-request oracle cycles spread over every host core this
    process may run on (os.sched_getaffinity), one OS thread per core; each
    oracle call is single-threaded C and releases the GIL, so the threads run
    in parallel.  Rounds of one request per thread run until about `seconds`
    of wall time; the value is committed tokens over the wall time of the
    oracle's phases (draft + schedule + pack, then verify), the target
    stand-in between them excluded."""
    from concurrent.futures import ThreadPoolExecutor

    inp = host_inputs(inp)
    n_thr = threads or host_cores()
    spent, toks, n = 0.0, 0, 0
    with ThreadPoolExecutor(max_workers=n_thr) as ex:
        while n < w.R and (spent < seconds or n == 0):
            idx = list(range(n, min(w.R, n + n_thr)))
            t0 = time.perf_counter()
            states = list(ex.map(lambda i: oracle_front(w, inp, [i], 0, dynamic, tau), idx))
            t1 = time.perf_counter()
            for st in states:
                oracle_target(w, st)
            t2 = time.perf_counter()
            toks += sum(ex.map(lambda st: oracle_back(w, st, observe), states))
            t3 = time.perf_counter()
            spent += (t1 - t0) + (t3 - t2)
            n += len(idx)
    return {"value": toks / spent, "unit": UNIT, "cores": n_thr, "kind": "oracle",
            "sample": f"{n} of {w.R} requests of one cycle, one per thread at a time on {n_thr} threads "
                      f"(os.sched_getaffinity), {spent:.1f} s wall"}


def run_reference(args, w):
    """The reference arm: the oracle as it stands, on the host cores.  Every
    step is one round of single-request oracle cycles, one per host core
    (os.sched_getaffinity) on its own thread, timed by the wall clock of the
    oracle's phases; the single-threaded rate on a bounded sample is
    reported beside it."""
    from concurrent.futures import ThreadPoolExecutor

    from speculative_decoding_markov_gb300 import synthetic

    inp = synthetic.generate(w, seed=0, device="cpu")
    if args.head == "rnn" and w.decode != "tree":
        inp.update(synthetic.rnn_inputs(w, seed=0))
    dynamic = args.scheduler == "dynamic" and w.decode != "tree"
    observe = args.observe and w.decode != "tree"
    tau = args.tau if args.scheduler == "threshold" and w.decode != "tree" else None
    hinp = host_inputs(inp)
    n_thr = host_cores()
    spent, toks, nxt = 0.0, 0, 0
    with ThreadPoolExecutor(max_workers=n_thr) as ex:
        for k in range(args.warmup + args.steps):
            idx = [(nxt + j) % w.R for j in range(n_thr)]
            nxt = (nxt + n_thr) % w.R
            t0 = time.perf_counter()
            states = list(ex.map(lambda i: oracle_front(w, hinp, [i], 0, dynamic, tau), idx))
            t1 = time.perf_counter()
            for st in states:
                oracle_target(w, st)
            t2 = time.perf_counter()
            c = sum(ex.map(lambda st: oracle_back(w, st, observe), states))
            t3 = time.perf_counter()
            if k >= args.warmup:
                spent += (t1 - t0) + (t3 - t2)
                toks += c
    value = toks / spent
    single = oracle_sample(w, inp, min(args.cpu_seconds, 10.0), dynamic, observe, tau)
    sample = (f"{n_thr} requests per step, one per thread on {n_thr} host threads (os.sched_getaffinity), "
              f"each a single-request oracle cycle (schedule over all {w.R}); wall clock of the oracle's phases")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": spent / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "value_counts": VALUE_COUNTS,
            "config": {"workload": w.name, "R": w.R, "B": w.B, "V": w.V, "r": w.r, "decode": w.decode,
                       "mode": w.modes[0], "scheduler": None if w.decode == "tree" else args.scheduler,
                       "tau": tau, "observe": observe, "head": None if w.decode == "tree" else args.head},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n_thr, "kind": "oracle", "sample": sample,
                             "single_thread": single},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def merge_ranks(t_local, units_local, world):
    """Whole-job figures of independent replicas: the slowest rank's timed
    seconds and the units (tokens, rows) summed over all ranks.  Host scalars
    only; the replicas exchange no data."""
    if world == 1:
        return t_local, list(units_local)
    import torch
    import torch.distributed as dist
    t = torch.tensor([t_local], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    u = torch.tensor(list(units_local), dtype=torch.float64)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), [float(x) for x in u.tolist()]


def other_workloads(args, world, rank, local):
    """The other four workloads, each in its own shorter run (the same
    timing, L2 flush and CUDA graphs; no host-copy leg; a bounded oracle
    sample on one core and on all cores)."""
    import gc

    import torch

    from speculative_decoding_markov_gb300.workloads import WORKLOADS

    res = {}
    for name in OTHER_WORKLOADS:
        a = argparse.Namespace(**vars(args))
        a.workload, a.steps, a.warmup = name, args.workload_steps, max(3, min(args.warmup, 10))
        a.no_e2e = True
        a.cpu_seconds = a.cpu_threads_seconds = min(args.cpu_seconds, 5.0)
        r = run_ours(a, WORKLOADS[name], world, rank, local)
        res[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "breakdown_ms_per_step",
                                       "tokens_per_step", "verified_rows_per_s", "roofline", "gpu_launches",
                                       "device_status", "clocks", "config") if k in r}
        if "cpu_baseline" in r:
            res[name]["cpu_baseline"] = r["cpu_baseline"]
        del r
        gc.collect()
        torch.cuda.empty_cache()
    return res


def main():
    args = parse()
    world, rank, local = dist_env()
    from speculative_decoding_markov_gb300.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.requests > 0:
        from speculative_decoding_markov_gb300.workloads import scaled
        w = scaled(w, R=args.requests)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)))
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    import __graft_entry__
    __graft_entry__.build()
    out = run_ours(args, w, world, rank, local)
    default_run = (args.workload == "qwen3_8b_chain" and args.requests == 0 and args.scheduler == "budget"
                   and args.head == "markov" and not args.observe)
    if default_run and not args.no_workloads and world == 1:
        out["workloads"] = other_workloads(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
