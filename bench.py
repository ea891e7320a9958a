"""Benchmark of the fused small-M MoE decode layer on one GB300 (or N replicas).

One step = one call of moe_decode_layer (router, top-k, gate/up + SwiGLU,
down + combine, shared expert) on one batch of M tokens. Weights are cold:
steps rotate over several seeded layer copies whose total size is far above
the 129 MB L2, so every step streams its experts from HBM. Inputs are seeded
synthetic data (moe_decode_gb300.synth); nothing is read from disk.

Headline line: Ling-shape layer (H=2560, E=512, top-8, I=768, one shared
expert), bf16 weights, M=1, 4 rotated layer copies. The other workloads
(M=6 independent tokens, M=10 with ~50% consecutive overlap, MXFP4 experts at
M=1 and M=6) are measured in the same run and reported under "also".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE decode layer µs/step and achieved HBM GB/s (cold weights) at M=1/6/10"
PERIOD = 64  # input ring length; the copy rotation divides it

WORKLOADS = {
    "ling_m1": dict(M=1, wfmt=0, copies=4, gen="independent"),
    "ling_m6": dict(M=6, wfmt=0, copies=4, gen="independent"),
    "ling_m10": dict(M=10, wfmt=0, copies=4, gen="overlap"),
    "mxfp4_m1": dict(M=1, wfmt=1, copies=8, gen="independent"),
    "mxfp4_m6": dict(M=6, wfmt=1, copies=8, gen="independent"),
    "fp8_m1": dict(M=1, wfmt=2, copies=6, gen="independent"),
    "fp8_m6": dict(M=6, wfmt=2, copies=6, gen="independent"),
    # small case for detailed profiler captures: the Ling layer cut to 128
    # experts (1.5 GB per copy), still far above L2
    "ling_e128_m1": dict(M=1, wfmt=0, copies=2, gen="independent", E=128),
    "mxfp4_e128_m6": dict(M=6, wfmt=1, copies=2, gen="independent", E=128),
}


# output layer (lm_head): the model's 157,184 x 2,560 vocabulary matrix (805 MB
# in bf16, already far above L2: one copy is cold at every step)
LM_WORKLOADS = {
    "lmhead_bf16_m1": dict(M=1, wfmt=0, V=157184, H=2560),
    "lmhead_fp8_m1": dict(M=1, wfmt=2, V=157184, H=2560),
    "lmhead_bf16_m6": dict(M=6, wfmt=0, V=157184, H=2560),
}


def layer_shape(name: str):
    from moe_decode_gb300 import synth
    E = WORKLOADS[name].get("E", synth.LING.n_experts)
    return synth.LayerShape(synth.LING.hidden, E, synth.LING.top_k, synth.LING.inter, synth.LING.shared_inter)


def describe(name: str) -> str:
    w = WORKLOADS[name]
    E = w.get("E", 512)
    fmt = {0: "bf16", 1: "MXFP4 (e2m1 + e8m0/32) routed experts, bf16 router and shared expert",
           2: "FP8 (e4m3 + fp32 scale/128) routed experts, bf16 router and shared expert"}[w["wfmt"]]
    gen = ("tokens drawn independently" if w["gen"] == "independent"
           else "tokens with ~50% consecutive top-8 overlap")
    return (f"Ling-shape MoE layer H=2560 E={E} top-8 I=768 shared I=768, {fmt}, M={w['M']} ({gen}), "
            f"cold weights rotated over {w['copies']} layer copies")


# ----------------------------------------------------------------------------- helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    rec = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            rec[k.strip()] = v.strip().strip("`")
    try:
        if rec.get("kernel_source_sha256") != kernel_source_sha():
            return None
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def kernel_source_sha() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed
    region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def visible_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v for v in vis.split(",") if v.strip()]
        try:
            return int(ids[local_rank])
        except (ValueError, IndexError):
            return local_rank
    return local_rank


# ----------------------------------------------------------------------------- our arm

class Workload:
    def __init__(self, name: str, device):
        from moe_decode_gb300 import api, synth
        self.api, self.synth = api, synth
        self.name = name
        w = WORKLOADS[name]
        self.M, self.wfmt, self.ncopy = w["M"], w["wfmt"], w["copies"]
        sh = layer_shape(name)
        self.shape = sh
        self.cshape = api.make_shape(sh.hidden, sh.n_experts, sh.top_k, sh.inter, sh.shared_inter, self.wfmt)
        self.layers = [synth.device_layer(sh, c, self.wfmt, device) for c in range(self.ncopy)]
        self.weights = [api.ExpertWeights(w1=L["w1"], w3=L["w3"], w2=L["w2"], ws1=L["ws1"], ws3=L["ws3"],
                                          ws2=L["ws2"], s1=L.get("s1"), s3=L.get("s3"), s2=L.get("s2"))
                        for L in self.layers]
        self.cweights = [wt.cstruct() for wt in self.weights]
        gen = synth.x_independent if w["gen"] == "independent" else synth.x_overlap
        self.xs = torch.stack([gen(sh, s, self.M, device=device) for s in range(PERIOD)])
        self.ws = api.workspace(self.cshape, self.M)
        self.y = torch.empty((self.M, sh.hidden), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((PERIOD, self.M, sh.top_k), dtype=torch.int32, device=device)
        self.wout = torch.empty((PERIOD, self.M, sh.top_k), dtype=torch.float32, device=device)
        self.weight_bytes = sum(t.numel() * t.element_size() for L in self.layers for t in L.values())

    def step(self, s: int, stream, idx=None, w=None, x=None, y=None):
        c = s % self.ncopy
        L = self.layers[c]
        self.api.decode_layer(self.xs[s % PERIOD] if x is None else x, L["Wg"], self.weights[c], self.cshape,
                              self.y if y is None else y, self.ws, idx, w, stream=stream,
                              cweights=self.cweights[c])

    def routing_pass(self, stream):
        """One untimed pass over the period to record the routing of every
        step (for the algorithmic byte count)."""
        for s in range(PERIOD):
            self.step(s, stream, self.idx[s], self.wout[s])
        stream.synchronize()
        st = self.api.read_status(self.ws, stream)
        if st != 0:
            raise RuntimeError(f"device status {st}")
        idx = self.idx.cpu().numpy()
        self.distinct = np.array([len(np.unique(idx[s])) for s in range(PERIOD)])

    def step_bytes(self, s: int) -> float:
        """Algorithmic HBM bytes of step s: router + touched experts + shared
        expert + x in + y out + routing out."""
        sh = self.shape
        H, I, E = sh.hidden, sh.inter, sh.n_experts
        U = int(self.distinct[s % PERIOD])
        if self.wfmt == 0:
            expert = 3 * H * I * 2
        elif self.wfmt == 1:
            expert = 2 * (I * H // 2 + I * H // 32) + (H * I // 2 + H * I // 32)
        else:
            expert = 3 * (H * I + H * I // 128 * 4)
        shared = 3 * H * sh.shared_inter * 2
        return E * H * 2 + U * expert + shared + 2 * self.M * H * 2 + self.M * sh.top_k * 8

    def mean_bytes(self, K: int) -> float:
        return sum(self.step_bytes(s) for s in range(K)) / K


class LmWorkload:
    """Output-layer GEMV: logits [M, V] of M tokens (one launch per step)."""

    def __init__(self, name: str, device):
        from moe_decode_gb300 import api, synth
        self.api = api
        self.name = name
        w = LM_WORKLOADS[name]
        self.M, self.wfmt, self.V, self.H = w["M"], w["wfmt"], w["V"], w["H"]
        Wb = synth.normal_bf16(3000, 1, 0, self.V * self.H, synth.WEIGHT_SIGMA, device).view(self.V, self.H)
        if self.wfmt == 0:
            self.W, self.scale = Wb, None
        else:
            self.W = torch.empty((self.V, self.H), dtype=torch.uint8, device=device)
            self.scale = torch.empty((self.V, 1), dtype=torch.float32, device=device)
            api.fp8_quantize(Wb, self.H, self.W, self.scale)
            del Wb
        self.xs = torch.stack([synth.x_independent(synth.LING, s, self.M, device=device) for s in range(PERIOD)])
        self.logits = torch.empty((self.M, self.V), dtype=torch.float32, device=device)
        self.ws = torch.empty(api.LM_HEAD_WORKSPACE_BYTES, dtype=torch.uint8, device=device)
        api.workspace_init(self.ws)
        self.weight_bytes = self.W.numel() * self.W.element_size()
        self.distinct = np.zeros(1)

    def step(self, s: int, stream, idx=None, w=None, x=None, y=None):
        self.api.lm_head(self.xs[s % PERIOD] if x is None else x, self.W, self.V, self.H, self.logits, self.ws,
                         wfmt=self.wfmt, w_scale=None if self.scale is None else self.scale.view(-1), stream=stream)

    def routing_pass(self, stream):
        self.step(0, stream)
        stream.synchronize()

    def mean_bytes(self, K: int) -> float:
        """Weights (+ e4m3 row scales), tokens in, logits out."""
        return self.weight_bytes + (self.V * 4 if self.wfmt else 0) + self.M * self.H * 2 + self.M * self.V * 4


def capture_graph(wl: Workload, start: int, n: int, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        g.capture_begin()
        try:
            for s in range(start, start + n):
                wl.step(s, stream)
        finally:
            g.capture_end()
    return g


def time_device(wl: Workload, K: int, W: int, stream, use_graph: bool, dist_barrier, sampler=None):
    """Returns (elapsed_ms of exactly K steps, launch mode)."""
    mode = "stream"
    graphs = None
    if use_graph:
        try:
            n = min(PERIOD, K)
            full = capture_graph(wl, 0, n, stream)
            rem = K % n
            tail = capture_graph(wl, 0, rem, stream) if rem else None
            graphs = (full, K // n, tail, n)
            mode = "cuda-graph"
        except Exception as e:  # capture not supported: plain stream launches
            torch.cuda.synchronize()
            print(f"# graph capture failed ({e}); timing stream launches", file=sys.stderr)
            graphs = None
    for s in range(W):
        wl.step(s, stream)
    if graphs:
        graphs[0].replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    dist_barrier()
    torch.cuda.synchronize()
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        # NVTX range "timed_region": lets a profiler's launch list cover
        # exactly the timed steps (ncu --nvtx --nvtx-include timed_region/)
        torch.cuda.nvtx.range_push("timed_region")
        e0.record(stream)
        if graphs:
            full, reps, tail, n = graphs
            with torch.cuda.stream(stream):
                for _ in range(reps):
                    full.replay()
                if tail is not None:
                    tail.replay()
        else:
            for s in range(K):
                wl.step(s, stream)
        e1.record(stream)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
    dist_barrier()
    return e0.elapsed_time(e1), mode


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        pass


def time_e2e(wl: Workload, K: int, stream, zero_copy: bool):
    """Same metric through the public API with host buffers, the tokens of
    each step in pinned host memory and y read back to pinned host memory.
    zero_copy: the host buffers are handed to the call itself, and the
    kernel reads the tokens from, and writes y to, host memory over the
    coherent CPU-GPU link (no copy launches); otherwise each step issues a
    host->device copy of its tokens and a device->host copy of y around the
    call."""
    xh = wl.xs.cpu().pin_memory()
    yh = torch.empty_like(wl.y, device="cpu").pin_memory()
    xd = torch.empty_like(wl.xs[0])

    def one(s):
        if zero_copy:
            wl.step(s, stream, x=xh[s % PERIOD], y=yh)
        else:
            xd.copy_(xh[s % PERIOD], non_blocking=True)
            wl.step(s, stream, x=xd)
            yh.copy_(wl.y, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(8):
            one(s)
    torch.cuda.synchronize()
    graphs = None
    if zero_copy:
        # the steps replayed as CUDA graphs, as in the device timing: each
        # replay's kernels still read and write the host buffers
        try:
            n = min(PERIOD, K)
            gs = []
            for cnt in (n, K % n):
                if cnt == 0:
                    gs.append(None)
                    continue
                g = torch.cuda.CUDAGraph()
                with torch.cuda.stream(stream):
                    g.capture_begin()
                    try:
                        for s in range(cnt):
                            one(s)
                    finally:
                        g.capture_end()
                gs.append(g)
            graphs = (gs[0], K // n, gs[1])
            graphs[0].replay()
            torch.cuda.synchronize()
        except Exception as e:
            torch.cuda.synchronize()
            print(f"# e2e graph capture failed ({e}); timing stream launches", file=sys.stderr)
            graphs = None
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        if graphs:
            full, reps, tail = graphs
            for _ in range(reps):
                full.replay()
            if tail is not None:
                tail.replay()
        else:
            for s in range(K):
                one(s)
        e1.record(stream)
    torch.cuda.synchronize()
    if zero_copy:  # the host copy of y is the device result of the last step
        wl.step((K - 1) % PERIOD, stream, x=xh[(K - 1) % PERIOD])
        stream.synchronize()
        if not torch.equal(yh, wl.y.cpu()):
            raise RuntimeError("zero-copy result differs from the device-buffer result")
    ms = e0.elapsed_time(e1)
    return ms, xh[0].numel() * xh.element_size(), yh.numel() * yh.element_size()


def cpu_steps_for(name: str) -> int:
    """Oracle steps that make about 12 s of single-thread work (the oracle
    takes ~65 ms per Ling token on a Grace core; MXFP4 decode adds ~40%)."""
    w = WORKLOADS[name]
    per_step_s = 0.065 * w["M"] * (1.4 if w["wfmt"] else 1.0) * w.get("E", 512) / 512
    return max(1, int(12.0 / per_step_s))


def oracle_sample(wl: Workload, nsteps: int):
    """Times the CPU oracle (as it stands, one host thread) on `nsteps` steps
    of the workload. Each step's host copies of its touched experts are made
    before that step's clock starts; only the oracle calls are timed.
    Returns us per step."""
    import oracle
    oracle.build()
    sh, synth = wl.shape, wl.synth
    idx_all = wl.idx.cpu().numpy()
    shared = [tuple(synth.to_u16(L[n]) for n in ("ws1", "ws3", "ws2")) for L in wl.layers]
    Wg = [synth.to_u16(L["Wg"]) for L in wl.layers]
    dt = 0.0
    for s in range(nsteps):
        c = s % wl.ncopy
        L = wl.layers[c]
        x = synth.to_u16(wl.xs[s % PERIOD])
        experts = {int(e): synth.host_expert(sh, L, int(e), wl.wfmt) for e in np.unique(idx_all[s % PERIOD])}
        t0 = time.perf_counter()
        idx, w, _ = oracle.route(x, Wg[c], sh.top_k)
        missing = [int(e) for e in np.unique(idx) if int(e) not in experts]
        if missing:
            raise RuntimeError(f"oracle routed to experts {missing} the device did not")
        oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, shared[c], wfmt=wl.wfmt)
        dt += time.perf_counter() - t0
    return dt / nsteps * 1e6


def replica_timing(ms_local: float, K: int, world: int, device=None):
    """(job us per step, replica us per step). Every rank runs its own replica
    of the layer (the path has no exchange step), so the job's timed region is
    the slowest rank's (max over ranks) and N replicas complete N steps in it."""
    ms = ms_local
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    us_rep = ms * 1e3 / K
    return us_rep / world, us_rep


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="ling_m1")
    ap.add_argument("--also", default="ling_m6,ling_m10,mxfp4_m1,mxfp4_m6,fp8_m1,fp8_m6,"
                                      "lmhead_bf16_m1,lmhead_fp8_m1,lmhead_bf16_m6",
                    help="comma-separated extra workloads measured in the same run ('' for none)")
    ap.add_argument("--cpu-steps", type=int, default=0,
                    help="oracle steps timed for cpu_baseline (0: about 12 s of oracle work for the workload)")
    ap.add_argument("--no-graph", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local_rank)
        import torch.distributed as dist
        dist.init_process_group("nccl")

        def barrier():
            dist.barrier()
    else:
        def barrier():
            pass

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    from moe_decode_gb300 import build
    build.build()
    device = torch.device("cuda", local_rank if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)

    results = {}
    names = [args.workload] + [n for n in args.also.split(",") if n and n != args.workload]
    for name in names:
        wl = LmWorkload(name, device) if name in LM_WORKLOADS else Workload(name, device)
        wl.routing_pass(stream)
        main_run = name == args.workload
        sampler = ClockSampler(visible_gpu_index(local_rank)) if main_run else None
        K = args.steps if main_run else min(args.steps, 4096)
        ms, mode = time_device(wl, K, args.warmup, stream, not args.no_graph, barrier, sampler)
        st = wl.api.read_status(wl.ws, stream)
        if st != 0:
            raise RuntimeError(f"{name}: device status {st}")
        us_job, us_step = replica_timing(ms, K, world, device)
        nbytes = wl.mean_bytes(K)
        res = {"us_per_step": us_job, "us_per_step_per_replica": us_step,
               "hbm_gbs": nbytes / (us_step * 1e-6) / 1e9, "bytes_per_step": nbytes,
               "distinct_experts_mean": float(np.mean(wl.distinct)), "steps": K, "launch": mode,
               "weights_gb": wl.weight_bytes / 1e9}
        if main_run:
            res["clocks"] = sampler.summary()
            e2e_ms, h2d, d2h = time_e2e(wl, K, stream, zero_copy=True)
            e2c_ms, _, _ = time_e2e(wl, K, stream, zero_copy=False)
            res["e2e"] = {"value": e2e_ms * 1e3 / K, "unit": "us/step", "h2d_bytes_per_step": h2d,
                          "d2h_bytes_per_step": d2h,
                          "mode": "zero-copy: the call gets the pinned host buffers; the kernel reads the tokens "
                                  "and writes y over the coherent CPU-GPU link (steps replayed as CUDA graphs)",
                          "explicit_copies_us_per_step": e2c_ms * 1e3 / K}
            if rank == 0:
                res["cpu_steps"] = args.cpu_steps or cpu_steps_for(name)
                res["cpu_us"] = oracle_sample(wl, res["cpu_steps"])
        results[name] = res
        del wl
        torch.cuda.empty_cache()

    if rank != 0:
        return
    main_res = results[args.workload]
    peak, peak_kind = measured_peaks()
    achieved = main_res["hbm_gbs"]
    w = WORKLOADS[args.workload]
    traffic = traffic_record("moe_layer_kernel", args.workload)
    line = {
        "metric": METRIC,
        "value": round(main_res["us_per_step"], 3),
        "unit": "us/step",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": main_res["us_per_step"] / 1e3,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": {0: "bf16", 1: "mxfp4-weights/bf16-act", 2: "fp8-e4m3-weights/bf16-act"}[w["wfmt"]],
        "data": "synthetic (seeded counter-hash generator; N(0,0.02)-like weights, N(0,1)-like tokens)",
        "config": {"workload": describe(args.workload), "M": w["M"], "hidden": 2560,
                   "n_experts": w.get("E", 512),
                   "top_k": 8, "inter": 768, "shared_inter": 768, "layer_copies": w["copies"],
                   "weights_gb": round(main_res["weights_gb"], 2),
                   "l2": "inputs larger than L2 (layer copies rotated every step)",
                   "launch": main_res["launch"], "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "distinct_experts_mean": main_res["distinct_experts_mean"]},
        "hbm_gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "kernel": "moe_layer_kernel", "traffic": traffic},
        "cpu_baseline": {"value": round(main_res["cpu_us"], 1), "unit": "us/step", "cores": 1,
                         "kind": "oracle",
                         "sample": f"{main_res['cpu_steps']} steps of the same workload (same inputs, routing "
                                   f"and touched experts), oracle in one host thread"},
        "e2e": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in main_res["e2e"].items()},
        "gpu_launches": args.steps,
        "clocks": main_res["clocks"],
        "also": {n: {k: (round(v, 3) if isinstance(v, float) else v) for k, v in r.items()
                     if k in ("us_per_step", "hbm_gbs", "distinct_experts_mean", "steps", "launch")}
                 | {"roofline_frac": round(r["hbm_gbs"] / peak, 4)}
                 for n, r in results.items() if n != args.workload},
    }
    print(json.dumps(line))


def run_reference(args, rank: int, world: int):
    """The reference arm: the CPU oracle, as it stands, on the host cores, on
    the same workload (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from moe_decode_gb300 import synth
    oracle.build()
    w = WORKLOADS[args.workload]
    sh = layer_shape(args.workload)
    nsteps = max(1, min(args.steps, args.cpu_steps or cpu_steps_for(args.workload)))
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    gen = synth.x_independent if w["gen"] == "independent" else synth.x_overlap
    copies = {}
    wsteps = min(args.warmup, 3)

    def prepare(s):
        """Inputs of step s and host copies of the experts it touches."""
        c = s % w["copies"]
        if c not in copies:
            copies[c] = (synth.to_u16(synth.router_weight(sh, c, dev)),
                         tuple(synth.to_u16(m) for m in synth.shared_weights(sh, c, dev)))
        x = synth.to_u16(gen(sh, s % PERIOD, w["M"], device=dev))
        idx, _, _ = oracle.route(x, copies[c][0], sh.top_k)
        experts = {}
        for e in np.unique(idx):
            mats = synth.expert_weights(sh, c, int(e), dev)
            if w["wfmt"] == 0:
                experts[int(e)] = tuple(synth.to_u16(m) for m in mats)
            else:
                q = [synth.mxfp4_quantize(m) if w["wfmt"] == 1 else synth.fp8_quantize(m) for m in mats]
                experts[int(e)] = (q[0][0].cpu().numpy(), q[0][1].cpu().numpy(), q[1][0].cpu().numpy(),
                                   q[1][1].cpu().numpy(), q[2][0].cpu().numpy(), q[2][1].cpu().numpy())
        return x, copies[c][0], experts, copies[c][1]

    def run(job):
        x, Wg, experts, shared = job
        idx, wt, _ = oracle.route(x, Wg, sh.top_k)
        oracle.ffn(x, idx, wt, experts, sh.n_experts, sh.inter, shared, wfmt=w["wfmt"])

    # each step's inputs are prepared untimed, then the oracle's step is timed
    dt = 0.0
    for s in range(wsteps + nsteps):
        job = prepare(s)
        t0 = time.perf_counter()
        run(job)
        if s >= wsteps:
            dt += time.perf_counter() - t0
    us = dt / nsteps * 1e6
    sample = (f"{nsteps} of the requested {args.steps} steps timed (bounded sample), after "
              f"{wsteps} warm-up steps; oracle in one host thread")
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": "us/step", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32-accumulate (oracle)", "data": "synthetic",
            "config": {"workload": describe(args.workload), "M": w["M"]},
            "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
