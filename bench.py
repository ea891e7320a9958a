"""Benchmark of the fused small-M MoE decode layer on one GB300 (or N replicas).

One step = one call of moe_decode_layer (router, top-k, gate/up + SwiGLU,
down + combine, shared expert) on one batch of M tokens. Weights are cold:
steps rotate over several seeded layer copies whose total size is far above
the 129 MB L2, so every step streams its experts from HBM. Inputs are seeded
synthetic data (moe_decode_gb300.synth); nothing is read from disk.

Headline line: Ling-shape layer (H=2560, E=512, top-8, I=768, one shared
expert), bf16 weights, M=1. The number of rotated layer copies is derived
from the device's L2 size: a copy is reused only after more than 3 x L2 bytes
of other copies' weights were streamed (checked after the routing pass). The
other workloads (M=6 independent tokens, M=10 with ~50% consecutive overlap,
the M=1..16 verify-length sweep, MXFP4 and FP8 experts at M=1 and M=6, the
output layer) are measured in the same run and reported under "also".

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

# copies: layer copies rotated per step. The full-size workloads use at least
# as many as the cold-weight rule needs (see cold_copies); the small profiling
# cases keep a fixed, small count.
# down_t: the layer is given its down projections also transposed (made once
# at load time with moe_transpose_down), which one-token calls use to split the
# down projection along the intermediate dimension (no grid barrier between
# the gate/up and down projections; measured slower than the two-phase layer
# at the Ling shape, reported beside it)
WORKLOADS = {
    "ling_m1": dict(M=1, wfmt=0, copies=4, gen="independent"),
    "ling_m1_splitk": dict(M=1, wfmt=0, copies=4, gen="independent", down_t=True),
    "ling_m6": dict(M=6, wfmt=0, copies=4, gen="independent"),
    "ling_m10": dict(M=10, wfmt=0, copies=4, gen="overlap"),
    "mxfp4_m1": dict(M=1, wfmt=1, copies=8, gen="independent"),
    "mxfp4_m6": dict(M=6, wfmt=1, copies=8, gen="independent"),
    "fp8_m1": dict(M=1, wfmt=2, copies=8, gen="independent"),
    "fp8_m6": dict(M=6, wfmt=2, copies=8, gen="independent"),
    # small cases for detailed profiler captures: the Ling layer cut to 128
    # experts (1.5 GB per copy), still far above L2
    "ling_e128_m1": dict(M=1, wfmt=0, copies=2, gen="independent", E=128, fixed_copies=True),
    "ling_e128_m1_splitk": dict(M=1, wfmt=0, copies=2, gen="independent", E=128, fixed_copies=True, down_t=True),
    "ling_e128_m10": dict(M=10, wfmt=0, copies=2, gen="overlap", E=128, fixed_copies=True),
    "ling_e128_m16": dict(M=16, wfmt=0, copies=2, gen="overlap", E=128, fixed_copies=True),
    "mxfp4_e128_m6": dict(M=6, wfmt=1, copies=2, gen="independent", E=128, fixed_copies=True),
    "fp8_e128_m6": dict(M=6, wfmt=2, copies=2, gen="independent", E=128, fixed_copies=True),
}
# the verify-length sweep: M = 1..16 tokens with ~50% consecutive top-8 overlap
for _m in range(1, 17):
    WORKLOADS[f"sweep_m{_m}"] = dict(M=_m, wfmt=0, copies=4, gen="overlap")
SWEEP = ",".join(f"sweep_m{m}" for m in range(1, 17))


# output layer (lm_head): the model's 157,184 x 2,560 vocabulary matrix (805 MB
# in bf16, already far above L2: one copy is cold at every step)
LM_WORKLOADS = {
    "lmhead_bf16_m1": dict(M=1, wfmt=0, V=157184, H=2560),
    "lmhead_fp8_m1": dict(M=1, wfmt=2, V=157184, H=2560),
    "lmhead_bf16_m6": dict(M=6, wfmt=0, V=157184, H=2560),
    "lmhead_bf16_m2": dict(M=2, wfmt=0, V=157184, H=2560),
    "lmhead_bf16_m16": dict(M=16, wfmt=0, V=157184, H=2560),
}


def layer_shape(name: str):
    from moe_decode_gb300 import synth
    E = WORKLOADS[name].get("E", synth.LING.n_experts)
    return synth.LayerShape(synth.LING.hidden, E, synth.LING.top_k, synth.LING.inter, synth.LING.shared_inter)


def expert_bytes(shape, wfmt: int) -> int:
    H, I = shape.hidden, shape.inter
    if wfmt == 0:
        return 3 * H * I * 2
    if wfmt == 1:
        return 2 * (I * H // 2 + I * H // 32) + (H * I // 2 + H * I // 32)
    return 3 * (H * I + H * I // 128 * 4)


def min_step_bytes(shape, wfmt: int, M: int) -> int:
    """Fewest algorithmic bytes a step can touch: the router, the shared
    expert and the k experts of one token (|U| >= k)."""
    return (shape.n_experts * shape.hidden * 2 + shape.top_k * expert_bytes(shape, wfmt)
            + 3 * shape.hidden * shape.shared_inter * 2 + 4 * M * shape.hidden)


def cold_copies(name: str, l2_bytes: int) -> int:
    """Layer copies rotated per step so that weights are cold: a copy is
    reused only after more than 3 x L2 bytes of other copies' weights were
    streamed. The count is a power of two (it divides the input ring)."""
    w = WORKLOADS[name]
    c = w["copies"]
    if w.get("fixed_copies"):
        return c
    need = 3 * l2_bytes / min_step_bytes(layer_shape(name), w["wfmt"], w["M"])
    while c - 1 <= need:
        c *= 2
    return c


def describe(name: str, copies: int) -> str:
    w = WORKLOADS[name]
    E = w.get("E", 512)
    fmt = {0: "bf16", 1: "MXFP4 (e2m1 + e8m0/32) routed experts, bf16 router and shared expert",
           2: "FP8 (e4m3 + fp32 scale/128) routed experts, bf16 router and shared expert"}[w["wfmt"]]
    if w.get("down_t"):
        fmt += " (down projections given transposed: split-K one-token path)"
    gen = ("tokens drawn independently" if w["gen"] == "independent"
           else "tokens with ~50% consecutive top-8 overlap")
    return (f"Ling-shape MoE layer H=2560 E={E} top-8 I=768 shared I=768, {fmt}, M={w['M']} ({gen}), "
            f"cold weights rotated over {copies} layer copies")


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
        # wait (at most 3 s) until the sampler is running
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < 3.0:
            time.sleep(0.01)
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

class LayerCache:
    """Device layer copies shared by the workloads of one run that use the
    same shape and weight format (the M sweep reuses one set)."""

    def __init__(self):
        self.sets = {}

    def get(self, sh, wfmt: int, copies: int, device):
        key = (sh, wfmt)
        have = self.sets.get(key, [])
        from moe_decode_gb300 import synth
        while len(have) < copies:
            have.append(synth.device_layer(sh, len(have), wfmt, device))
        self.sets[key] = have
        return have[:copies]

    def drop_except(self, keep_key=None):
        for k in list(self.sets):
            if k != keep_key:
                del self.sets[k]


class Workload:
    def __init__(self, name: str, device, cache: LayerCache, l2_bytes: int):
        from moe_decode_gb300 import api, synth
        self.api, self.synth = api, synth
        self.name = name
        w = WORKLOADS[name]
        self.M, self.wfmt = w["M"], w["wfmt"]
        self.ncopy = cold_copies(name, l2_bytes)
        sh = layer_shape(name)
        self.shape = sh
        self.cshape = api.make_shape(sh.hidden, sh.n_experts, sh.top_k, sh.inter, sh.shared_inter, self.wfmt)
        self.layers = cache.get(sh, self.wfmt, self.ncopy, device)
        self.down_t = bool(w.get("down_t"))
        if self.down_t:
            for L in self.layers:
                if "w2t" not in L:  # kept with the cached copy for later workloads
                    L["w2t"] = api.transpose_down(L["w2"])
                    L["ws2t"] = api.transpose_down(L["ws2"])
        used = ["Wg", "w1", "w3", "w2", "ws1", "ws3", "ws2", "s1", "s3", "s2"]
        if self.down_t:
            used = [n for n in used if n not in ("w2", "ws2")] + ["w2t", "ws2t"]
        self.weights = [api.ExpertWeights(w1=L["w1"], w3=L["w3"], w2=L["w2"], ws1=L["ws1"], ws3=L["ws3"],
                                          ws2=L["ws2"], s1=L.get("s1"), s3=L.get("s3"), s2=L.get("s2"),
                                          w2t=L.get("w2t") if self.down_t else None,
                                          ws2t=L.get("ws2t") if self.down_t else None)
                        for L in self.layers]
        self.used_keys = used
        self.cweights = [wt.cstruct() for wt in self.weights]
        gen = synth.x_independent if w["gen"] == "independent" else synth.x_overlap
        self.xs = torch.stack([gen(sh, s, self.M, device=device) for s in range(PERIOD)])
        self.ws = api.workspace(self.cshape, self.M)
        self.y = torch.empty((self.M, sh.hidden), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((PERIOD, self.M, sh.top_k), dtype=torch.int32, device=device)
        self.wout = torch.empty((PERIOD, self.M, sh.top_k), dtype=torch.float32, device=device)
        self.weight_bytes = sum(L[n].numel() * L[n].element_size() for L in self.layers for n in self.used_keys
                                if n in L)

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
        H, E = sh.hidden, sh.n_experts
        U = int(self.distinct[s % PERIOD])
        shared = 3 * H * sh.shared_inter * 2
        return E * H * 2 + U * expert_bytes(sh, self.wfmt) + shared + 2 * self.M * H * 2 + self.M * sh.top_k * 8

    def mean_bytes(self, K: int) -> float:
        return sum(self.step_bytes(s) for s in range(K)) / K

    def reuse_bytes_min(self) -> float:
        """Fewest weight bytes streamed between two uses of one copy: the
        other copies' steps in between (ncopy - 1 of them)."""
        per = sorted(self.step_bytes(s) for s in range(PERIOD))
        return float(sum(per[:self.ncopy - 1]))


class LmWorkload:
    """Output-layer GEMV: logits [M, V] of M tokens (one launch per step).
    Every step reads the whole matrix, so between two reads of a weight byte
    at least one full pass over its own copy is streamed; copies are added
    (rotated per step) until that exceeds 3 x L2."""

    def __init__(self, name: str, device, cache=None, l2_bytes: int = 0):
        from moe_decode_gb300 import api, synth
        self.api = api
        self.name = name
        w = LM_WORKLOADS[name]
        self.M, self.wfmt, self.V, self.H = w["M"], w["wfmt"], w["V"], w["H"]
        per_copy = self.V * self.H * (2 if self.wfmt == 0 else 1)
        self.ncopy = 1
        while self.ncopy * per_copy <= 3 * l2_bytes:
            self.ncopy *= 2
        self.W, self.scale = [], []
        for c in range(self.ncopy):
            Wb = synth.normal_bf16(3000 + c, 1, 0, self.V * self.H, synth.WEIGHT_SIGMA, device).view(self.V, self.H)
            if self.wfmt == 0:
                self.W.append(Wb)
                self.scale.append(None)
            else:
                q = torch.empty((self.V, self.H), dtype=torch.uint8, device=device)
                sc = torch.empty((self.V, 1), dtype=torch.float32, device=device)
                api.fp8_quantize(Wb, self.H, q, sc)
                del Wb
                self.W.append(q)
                self.scale.append(sc.view(-1))
        self.xs = torch.stack([synth.x_independent(synth.LING, s, self.M, device=device) for s in range(PERIOD)])
        self.logits = torch.empty((self.M, self.V), dtype=torch.float32, device=device)
        self.ws = torch.empty(api.LM_HEAD_WORKSPACE_BYTES, dtype=torch.uint8, device=device)
        api.workspace_init(self.ws)
        self.copy_bytes = per_copy
        self.weight_bytes = per_copy * self.ncopy
        self.distinct = np.zeros(1)

    def step(self, s: int, stream, idx=None, w=None, x=None, y=None):
        c = s % self.ncopy
        self.api.lm_head(self.xs[s % PERIOD] if x is None else x, self.W[c], self.V, self.H, self.logits, self.ws,
                         wfmt=self.wfmt, w_scale=self.scale[c], stream=stream)

    def routing_pass(self, stream):
        self.step(0, stream)
        stream.synchronize()

    def reuse_bytes_min(self) -> float:
        return float(self.ncopy * self.copy_bytes)

    def mean_bytes(self, K: int) -> float:
        """Weights (+ e4m3 row scales), tokens in, logits out."""
        return self.copy_bytes + (self.V * 4 if self.wfmt else 0) + self.M * self.H * 2 + self.M * self.V * 4


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
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        # the W warm-up steps (and one replay of the timed graph) run right
        # before the timed region, inside the clock sampler's context: an
        # idle GPU (e.g. while the sampler starts) would make the first
        # timed steps slower, which a short timed region cannot amortise
        for s in range(W):
            wl.step(s, stream)
        if graphs:
            with torch.cuda.stream(stream):
                graphs[0].replay()
        torch.cuda.synchronize()
        dist_barrier()
        torch.cuda.synchronize()
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


def oracle_sample(wl: Workload, nsteps: int, nthreads: int = 1):
    """Times the CPU oracle (as it stands) on `nsteps` steps of the workload:
    in one host thread (nthreads 1), or with its expert calls spread over
    host threads (0: all; the same arithmetic and bits). Each step's host
    copies of its touched experts are made before that step's clock starts;
    only the oracle calls are timed. Returns us per step."""
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
        oracle.ffn(x, idx, w, experts, sh.n_experts, sh.inter, shared[c], wfmt=wl.wfmt, nthreads=nthreads)
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
    ap.add_argument("--also", default="ling_m1_splitk,ling_m6,ling_m10,mxfp4_m1,mxfp4_m6,fp8_m1,fp8_m6,"
                                      "lmhead_bf16_m1,lmhead_fp8_m1,lmhead_bf16_m6," + SWEEP,
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
    l2_bytes = int(torch.cuda.get_device_properties(device).L2_cache_size)

    results = {}
    names = [args.workload] + [n for n in args.also.split(",") if n and n != args.workload]
    cache = LayerCache()
    for name in names:
        if name in LM_WORKLOADS:
            cache.drop_except()
            wl = LmWorkload(name, device, l2_bytes=l2_bytes)
        else:
            cache.drop_except((layer_shape(name), WORKLOADS[name]["wfmt"]))
            wl = Workload(name, device, cache, l2_bytes)
        wl.routing_pass(stream)
        # cold weights: a copy is reused only after > 3 x L2 bytes of others
        reuse = wl.reuse_bytes_min()
        if not WORKLOADS.get(name, {}).get("fixed_copies") and reuse <= 3 * l2_bytes:
            # (the profiling cases keep a small, fixed rotation on purpose)
            raise RuntimeError(f"{name}: only {reuse / 1e6:.0f} MB between reuses of a layer copy "
                               f"(<= 3 x L2 = {3 * l2_bytes / 1e6:.0f} MB)")
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
               "weights_gb": wl.weight_bytes / 1e9, "copies": wl.ncopy, "reuse_bytes_min": reuse}
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
                import oracle
                res["cpu_steps"] = args.cpu_steps or cpu_steps_for(name)
                res["cpu_us"] = oracle_sample(wl, res["cpu_steps"])
                res["cpu_all_us"] = oracle_sample(wl, res["cpu_steps"], nthreads=0)
                res["cpu_threads"] = oracle.threads()
        results[name] = res
        del wl
        torch.cuda.empty_cache()
    cache.drop_except()

    if rank != 0:
        return
    main_res = results[args.workload]
    peak, peak_kind = measured_peaks()
    achieved = main_res["hbm_gbs"]
    w = WORKLOADS[args.workload]
    kname = "moe_layer_splitk_kernel" if w.get("down_t") and w["M"] == 1 else "moe_layer_kernel"
    traffic = traffic_record(kname, args.workload)
    tasks = w["M"] * (layer_shape(args.workload).top_k + 1)
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
        "config": workload_config(args.workload, main_res["copies"], world, main_res, l2_bytes),
        "hbm_gbs": round(achieved, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                     "kernel": kname, "traffic": traffic},
        "cpu_baseline": {"value": round(main_res["cpu_us"], 1), "unit": "us/step", "cores": 1,
                         "kind": "oracle",
                         "sample": f"{main_res['cpu_steps']} steps of the same workload (same inputs, routing "
                                   f"and touched experts), oracle in one host thread",
                         "all_cores": {"value": round(main_res["cpu_all_us"], 1), "unit": "us/step",
                                       "cores": min(main_res["cpu_threads"], tasks),
                                       "host_cpus": os.cpu_count(), "threads_available": main_res["cpu_threads"],
                                       "sample": f"the same {main_res['cpu_steps']} steps; the oracle's "
                                                 f"{tasks} (token, expert) calls per step (the shared expert "
                                                 f"included) spread over OpenMP threads, same bits"}},
        "e2e": {k: (round(v, 3) if isinstance(v, float) else v) for k, v in main_res["e2e"].items()},
        "gpu_launches": args.steps,
        "clocks": main_res["clocks"],
        "also": {n: {k: (round(v, 3) if isinstance(v, float) else v) for k, v in r.items()
                     if k in ("us_per_step", "hbm_gbs", "distinct_experts_mean", "steps", "launch", "copies")}
                 | {"roofline_frac": round(r["hbm_gbs"] / peak, 4)}
                 for n, r in results.items() if n != args.workload},
    }
    print(json.dumps(line))


def workload_config(name: str, copies: int, world: int, res=None, l2_bytes: int = 0) -> dict:
    """The bench line's config for a layer workload (the same dict on the
    reference arm)."""
    w = WORKLOADS[name]
    cfg = {"workload": describe(name, copies), "M": w["M"], "hidden": 2560, "n_experts": w.get("E", 512),
           "top_k": 8, "inter": 768, "shared_inter": 768, "layer_copies": copies,
           "l2": "inputs larger than L2 (layer copies rotated every step)",
           "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}
    if res is not None:
        cfg["weights_gb"] = round(res["weights_gb"], 2)
        cfg["launch"] = res["launch"]
        cfg["distinct_experts_mean"] = res["distinct_experts_mean"]
        cfg["cold_weights"] = {"l2_bytes": l2_bytes, "bytes_between_reuses_min": int(res["reuse_bytes_min"]),
                               "rule": "bytes streamed between two uses of a layer copy > 3 x L2"}
    return cfg


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
    # the same layer-copy rotation as the GPU arm (it depends on the L2 size)
    l2_bytes = int(torch.cuda.get_device_properties(0).L2_cache_size) if dev == "cuda" else 126 << 20
    copies_ref = cold_copies(args.workload, l2_bytes)

    def prepare(s):
        """Inputs of step s and host copies of the experts it touches."""
        c = s % copies_ref
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
            "config": workload_config(args.workload, copies_ref, world),
            "cpu_baseline": {"value": round(us, 1), "unit": "us/step", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(us, 1), "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
