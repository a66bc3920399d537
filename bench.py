#!/usr/bin/env python3
"""Benchmark of the routed MoE expert-FFN layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_m1|tiny|sweep_m<M>[_zipf]|large_m1|large_m8|awq_fixture_a|awq_m1|probe_m16384]

A step is one pass of the hot path over one batch of fresh synthetic input:
top-k routing of the step's router logits, then the layer (at one token the
routing runs inside the layer's single kernel; the grouped path adds the
alignment).  The default workload is the 128-expert d=2048 / I=768 top-8
layer at M=1 with MXFP8 weights, fresh routing every step.

Timing: K steps run back to back in CUDA graphs, bracketed by one pair of
CUDA events on the launching stream, as a model runs its stack of MoE layers.
Each step reads the next of L copies of the layer's weights (16 at M=1, 10 GB)
with its own input, so its weights were last read L steps earlier: the inputs
of the timed steps are larger than the L2 and no flush is needed.  Also
reported: one isolated call (the L2 evicted by a 1 GiB read before it), the
layer call alone back to back (routing computed ahead of time) for the
roofline, and the end-to-end call through the public API with host buffers.

Metric: achieved HBM TB/s of the layer = algorithmic bytes (the distinct
routed experts' MXFP8 weights incl. scales, plus x, the router logits and y)
divided by the step time; also reported as microseconds per layer.

--impl reference times the CPU oracle (binary64, test infrastructure) on
the host cores on a bounded sample of the same workload, in the same units.
Multi-GPU (torchrun): independent replicas, one per GPU, no collective.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer µs & achieved HBM TB/s (% of GB300 peak) at M=1–64 decode"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 * 2 ** 20


# ------------------------------------------------------------------ helpers

def workload_from_name(name: str):
    from top_moe_expert_gb300 import inputs
    if name == "decode_m1":
        return inputs.DECODE
    if name == "tiny":
        return inputs.TINY
    if name == "large_m1":
        return inputs.LARGE_M1
    if name == "large_m8":
        return inputs.LARGE_M8
    if name == "awq_fixture_a":
        return inputs.AWQ_FIXTURE
    if name == "awq_m1":
        # one token of the fixture-A closed-form routing: 8 distinct experts
        return inputs.Workload("awq_m1_d2048_i768_e128_k8", M=1, d=2048, I=768, E=128, k=8, fmt="awq4",
                               routing="fixture_a", seed=3)
    if name == "probe_m16384":
        return inputs.Workload("grouped_probe_m16384_d2048_i768_e128_k8", M=16384, d=2048, I=768, E=128, k=8,
                               seed=2)
    if name.startswith("nv4_m"):
        # paired 4:8 sparse NVFP4 weights (random admissible packing) at the sweep's shapes
        M = int(name[len("nv4_m"):])
        return inputs.Workload(f"nv4_m{M}_uniform_d2048_i768_e128_k8", M=M, d=2048, I=768, E=128, k=8,
                               fmt="nvfp4s", seed=2)
    if name.startswith("sweep_m"):
        rest = name[len("sweep_m"):]
        routing = "zipf" if rest.endswith("_zipf") else "uniform"
        return inputs.sweep(int(rest.split("_")[0]), routing)
    raise SystemExit(f"unknown workload {name}")


def expert_bytes(wl, path: str = "decode") -> int:
    """Weight bytes of one expert.  MXFP8: 3*I*d codes + 3*I*d/32 scale
    bytes.  AWQ-4bit: 3*I*d/2 packed values + an fp16 scale and a 4-bit zero
    per 128 values.  NVFP4S: 3*I*d/4 bytes of kept codes, plus 3*I*d/16
    pattern and 3*I*d/32 scale bytes (decode path) or the grouped path's
    16-byte side record per 128 weights (3*I*d/8), plus the expert's two
    fp32 values: its constants of W13 and W2 (decode) or the two per-expert
    factors (grouped)."""
    n = 3 * wl.I * wl.d
    if wl.fmt == "awq4":
        return n // 2 + n // 128 * 2 + n // 128 // 2
    if wl.fmt == "nvfp4s":
        return n // 4 + (n // 8 if path == "grouped" else n // 16 + n // 32) + 8
    return n * 33 // 32


def layer_bytes(wl, ids: np.ndarray, path: str = "decode") -> int:
    """Algorithmic bytes of one layer call: distinct routed experts' weights,
    x and the routing (ids, weights) read, y written (bf16)."""
    distinct = len(np.unique(ids[(ids >= 0) & (ids < wl.E)]))
    return distinct * expert_bytes(wl, path) + wl.M * wl.d * 2 + wl.M * wl.k * 8 + wl.M * wl.d * 2


def step_bytes(wl, ids: np.ndarray, path: str = "decode") -> int:
    """Algorithmic bytes of one step: distinct routed experts' weights, the
    activations read (x, router logits) and the output written (bf16 y)."""
    distinct = len(np.unique(ids[(ids >= 0) & (ids < wl.E)]))
    routing = wl.M * wl.k * 8 if wl.routing == "fixture_a" else wl.M * wl.E * 4   # fixed ids/w, or logits
    return distinct * expert_bytes(wl, path) + wl.M * wl.d * 2 + routing + wl.M * wl.d * 2


def measured_mxfp8_tflops():
    """Dense MXFP8 tensor peak: the measured bf16 burst peak times the
    nominal fp8:bf16 ratio of 2 (4.5 vs 2.25 PFLOP/s)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return 2.0 * float(json.load(open(p))["bf16_tflops"]), "measured bf16 x 2"
    except Exception:
        return 2.0 * 1900.0, "fallback bf16 x 2"


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.perf_counter(), parts))

    def stop(self, t0: float, t1: float):
        """Summary of the samples that arrived inside [t0, t1] (the timed loop)."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        inside = [r for (t, r) in self.rows if t0 <= t <= t1]
        window = "inside the timed region"
        if not inside:
            # a timed region shorter than the sampling period: the samples
            # taken within 0.25 s of it (warm-up and the untimed steps around)
            inside = [r for (t, r) in self.rows if t0 - 0.25 <= t <= t1 + 0.25]
            window = "within 0.25 s of a timed region shorter than the sampling period"
        self.rows = inside
        if not self.rows:
            return None
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(self.rows), "window": window}


def committed_traffic(kernel_key: str, src_hash: str):
    """DRAM traffic per launch from the committed ncu summary, or None when the
    kernel sources changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        d = json.load(open(p))[kernel_key]
    except Exception:
        return None
    return d["bytes_per_launch"] if d.get("src_sha256") == src_hash else None


SRC_FILES = {
    "decode": ("decode.cu", "decode_pipe.cu", "pipe_common.cuh", "decode_stream.cu", "decode_internal.h", "topk.cu", "topk.cuh",
               "common.cuh", "tc.cuh", "attr.h"),
    "grouped": ("grouped.cu", "grouped_internal.h", "align.cu", "topk.cu", "topk.cuh", "common.cuh", "tc.cuh",
                "attr.h"),
    "awq": ("grouped_awq.cu", "grouped.cu", "grouped_internal.h", "align.cu", "common.cuh", "tc.cuh", "attr.h"),
    "awq_decode": ("decode.cu", "decode_pipe_awq.cu", "pipe_common.cuh", "decode_internal.h", "common.cuh", "tc.cuh",
                   "attr.h"),
    "nv4": ("grouped_awq.cu", "grouped.cu", "grouped_internal.h", "align.cu", "topk.cu", "topk.cuh", "common.cuh",
            "tc.cuh", "attr.h"),
    "nv4_decode": ("decode.cu", "decode_pipe_nv4.cu", "pipe_common.cuh", "decode_nvfp4s.cu", "nvfp4s.cuh",
                   "decode_internal.h", "topk.cu", "topk.cuh", "common.cuh", "tc.cuh", "attr.h"),
}


_C_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|//[^\n]*|/\*.*?\*/', re.S)


def code_only(text: str) -> str:
    """C/C++/CUDA source with its comments and blank lines removed (string
    and character literals kept), so that a comment edit leaves the hash of
    the compiled code unchanged."""
    text = _C_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def decode_src_hash(path: str = "decode") -> str:
    """SHA-256 over the kernel sources of one path, comments removed (the ncu
    counters in profiles/traffic.json are valid only for this code)."""
    h = hashlib.sha256()
    for f in SRC_FILES[path]:
        h.update(code_only(open(os.path.join(ROOT, "top_moe_expert_gb300", "csrc", f)).read()).encode())
    return h.hexdigest()


# ------------------------------------------------------------------ our arm

def grouped_block(wl) -> int:
    """MoE block size b of the grouped path: twice the expected rows per
    expert, rounded up to a power of two within [16, 128], so that most
    experts fit in one block and their weights stream once."""
    rows = max(1, 2 * wl.M * wl.k // wl.E)
    b = 16
    while b < rows and b < 128:
        b *= 2
    return b


def layer_copies(wl, step_bytes_est: int, layer_weight_bytes: int) -> int:
    """Copies of the layer's weights the timed steps rotate through (a model's
    stack of MoE layers): enough that a step's weights were last read at
    least 1.5 GB of other traffic ago (about 12 times the L2), at most 16
    copies and 48 GB."""
    want = -(-int(1.5e9) // max(1, step_bytes_est))
    cap = max(1, int(48e9 // max(1, layer_weight_bytes)))
    return max(1, min(16, want, cap))


class Step:
    """Device-resident workload: L copies of the layer's weights, a pool of
    fresh inputs (router logits, activations) and the buffers of one step.
    A step is top-k routing and the layer (decode path; at one token the
    routing runs inside the layer's kernel), or top-k, alignment and the
    grouped layer; with the fixed-routing AWQ workloads, the layer alone (with
    its alignment on the grouped path)."""

    def __init__(self, wl, n_inputs, device, path: str = "decode", block: int = 0, layers: int = 0):
        import top_moe_expert_gb300 as moe
        from top_moe_expert_gb300 import inputs
        self.moe, self.wl, self.dev, self.path = moe, wl, device, path
        self.awq = wl.fmt == "awq4"
        self.nv4 = wl.fmt == "nvfp4s"
        E, d, I, M, k = wl.E, wl.d, wl.I, wl.M, wl.k
        self.n_inputs = n_inputs
        # ---- layer 0's weights
        if self.awq:
            dev_t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)
            q13, s13, z13 = inputs.awq_weights(wl, "w13")
            q2, s2, z2 = inputs.awq_weights(wl, "w2")
            w0 = ((dev_t(q13), dev_t(s13).view(torch.float16), dev_t(z13)),
                  (dev_t(q2), dev_t(s2).view(torch.float16), dev_t(z2)))
            del q13, s13, z13, q2, s2, z2
        elif self.nv4:
            dev_t = lambda a: torch.from_numpy(a).to(device)
            v13, m13, c13, a13 = inputs.nvfp4s_weights(wl, "w13")
            v2, m2, c2, a2 = inputs.nvfp4s_weights(wl, "w2")
            w0 = ((dev_t(v13), dev_t(c13), dev_t(m13), dev_t(a13)), (dev_t(v2), dev_t(c2), dev_t(m2), dev_t(a2)))
            del v13, m13, c13, v2, m2, c2
        else:
            q13 = torch.empty((E, 2 * I, d), dtype=torch.uint8, device=device)
            s13 = torch.empty((E, 2 * I, d // 32), dtype=torch.uint8, device=device)
            q2 = torch.empty((E, d, I), dtype=torch.uint8, device=device)
            s2 = torch.empty((E, d, I // 32), dtype=torch.uint8, device=device)
            for e in range(E):
                moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w13", e, device), q13[e], s13[e])
                moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w2", e, device), q2[e], s2[e])
            w0 = ((q13, s13, None), (q2, s2, None))
        self.routed_in_layer = wl.fmt in ("mxfp8", "nvfp4s") and path == "decode" and M == 1 and E <= 768
        # one AWQ token: the layer is one kernel (the routing is fixed, so it is not in it)
        self.awq_pipe = self.awq and path == "decode" and M == 1
        lw_bytes = sum(t.numel() * t.element_size() for p in w0 for t in p if t is not None)
        self.ids_host = [self._host_ids(j) for j in range(n_inputs)]
        est = max(step_bytes(wl, ids, path) for ids in self.ids_host[:8])
        self.L = layers if layers > 0 else layer_copies(wl, est, lw_bytes)
        self.layer_weight_bytes = lw_bytes
        self.layers = []
        # NVFP4S grouped path: the layer's activation scales (constants of the
        # layer): alpha_x from the largest |x| of the inputs, alpha_h for |h|
        # up to 16 (the weights' RMS and N(0,1) inputs give |g|, |u| ~ 1)
        self.alpha_x = self.alpha_h = None
        for l in range(self.L):
            parts = w0 if l == 0 else tuple(tuple(t.clone() if t is not None else None for t in p) for p in w0)
            if self.nv4:
                (v13_, c13_, m13_, a13_), (v2_, c2_, m2_, a2_) = parts
                w13 = moe.Weights(moe.MOE_W_NVFP4S, v13_, c13_, m13_, a13_)
                w2 = moe.Weights(moe.MOE_W_NVFP4S, v2_, c2_, m2_, a2_)
                self.layers.append([w13, w2, (None, None)])
                continue
            (a13, b13, c13), (a2, b2, c2) = parts
            if self.awq:
                w13 = moe.Weights(moe.MOE_W_AWQ4, a13, b13, c13)
                w2 = moe.Weights(moe.MOE_W_AWQ4, a2, b2, c2)
            else:
                w13 = moe.Weights(moe.MOE_W_MXFP8, a13, b13)
                w2 = moe.Weights(moe.MOE_W_MXFP8, a2, b2)
            sfa = moe.moe_grouped_prepare(w13, w2) if (path == "grouped" and not self.awq) else (None, None)
            self.layers.append((w13, w2, sfa))
        del w0
        torch.cuda.empty_cache()
        # ---- inputs
        if self.awq:
            self.logits_host = torch.zeros((n_inputs, M, E), dtype=torch.float32)     # routing is fixed
            self.x_host = torch.stack([inputs.activations(wl, i, dtype=torch.float16) for i in range(n_inputs)])
        else:
            self.logits_host = torch.from_numpy(np.stack([inputs.router_logits(wl, i) for i in range(n_inputs)]))
            self.x_host = torch.stack([inputs.activations(wl, i) for i in range(n_inputs)])
        self.logits_all = self.logits_host.to(device)
        self.x_all = self.x_host.to(device)
        # x and the router logits share one device buffer, so an end-to-end
        # step's inputs arrive in one host-to-device copy
        xb = M * d * 2
        self.io = torch.empty(xb + (0 if self.awq else M * E * 4), dtype=torch.uint8, device=device)
        self.x = self.io[:xb].view(self.x_all.dtype).view(M, d)
        self.logits = (torch.empty((M, E), dtype=torch.float32, device=device) if self.awq
                       else self.io[xb:].view(torch.float32).view(M, E))
        if self.nv4 and path == "grouped":
            self.alpha_x = float(self.x_all.abs().max().item()) / (6 * 448)
            self.alpha_h = 16.0 / (6 * 448)
            for lay in self.layers:
                lay[2] = moe.moe_grouped_prepare_nvfp4s(lay[0], lay[1], self.alpha_x, self.alpha_h)
        self.layers = [tuple(l) for l in self.layers]
        self.io_host = ("x_host",) if self.awq else ("x_host", "logits_host")
        self.y = torch.empty((M, d), dtype=torch.bfloat16, device=device)
        if self.awq:
            fid = torch.from_numpy(inputs.fixture_a_ids(M, k, E)).to(device)
            fw = torch.from_numpy(inputs.fixture_a_weights(M, k, wl.seed)).to(device)
            self.ids, self.w = fid, fw
            self.ids_all = fid.expand(n_inputs, M, k)
            self.w_all = fw.expand(n_inputs, M, k)
        else:
            self.ids = torch.empty((M, k), dtype=torch.int32, device=device)
            self.w = torch.empty((M, k), dtype=torch.float32, device=device)
            # the routing of every input, for the layer-only timing
            self.ids_all = torch.empty((n_inputs, M, k), dtype=torch.int32, device=device)
            self.w_all = torch.empty((n_inputs, M, k), dtype=torch.float32, device=device)
            for j in range(n_inputs):
                moe.moe_topk_softmax(self.logits_all[j], k, self.ids_all[j], self.w_all[j])
        if path == "grouped":
            self.b = block or (wl.b if self.awq else grouped_block(wl))
            cr, cb = moe.moe_align_capacity(M, k, E, self.b)
            mk = lambda: (torch.empty(cr, dtype=torch.int32, device=device),
                          torch.empty(cb, dtype=torch.int32, device=device),
                          torch.empty(1, dtype=torch.int32, device=device))
            self.aligned = mk()
            na = moe.moe_align_workspace_size(M, k, E, self.b)
            self.ws_align = torch.empty(max(na, 256), dtype=torch.uint8, device=device) if na else None
            self.ws = torch.empty(moe.moe_ffn_grouped_workspace_size(M, k, d, I, self.b, cr), dtype=torch.uint8,
                                  device=device)
            # the alignment of every input (fixed routing: one), for the layer-only timing
            na_in = 1 if self.awq else n_inputs
            self.aligned_all = [mk() for _ in range(na_in)]
            for j in range(na_in):
                moe.moe_align_block_size(self.ids_all[j], E, self.b, out=self.aligned_all[j], ws=self.ws_align)
        else:
            self.b = 0
            self.ws = torch.zeros(moe.moe_ffn_decode_workspace_size(M, k, d, I), dtype=torch.uint8, device=device)
        self.stream = torch.cuda.Stream(device)
        torch.cuda.synchronize()

    def _host_ids(self, j: int) -> np.ndarray:
        from top_moe_expert_gb300 import inputs
        if self.awq:
            return inputs.fixture_a_ids(self.wl.M, self.wl.k, self.wl.E)
        return host_topk_ids(inputs.router_logits(self.wl, j), self.wl.k)

    def step_ids(self, i: int) -> np.ndarray:
        """Expert ids of step i (to count the distinct experts it reads)."""
        return self.ids_host[i % self.n_inputs]

    # ---- launches
    def launch_step(self, i: int, stream, x=None, logits=None):
        """Step i: input i mod n_inputs (or the given x / logits), layer i mod L."""
        moe, wl = self.moe, self.wl
        j, (w13, w2, (sfa13, sfa2)) = i % self.n_inputs, self.layers[i % self.L]
        x = self.x_all[j] if x is None else x
        logits = self.logits_all[j] if logits is None else logits
        if self.routed_in_layer:
            moe.moe_ffn_decode_logits(logits, x, wl.k, w13, w2, y=self.y, topk_ids=self.ids, topk_w=self.w,
                                      ws=self.ws, stream=stream)
            return
        if not self.awq:
            moe.moe_topk_softmax(logits, wl.k, self.ids, self.w, stream=stream)
        if self.path == "grouped":
            moe.moe_align_block_size(self.ids, wl.E, self.b, out=self.aligned, ws=self.ws_align, stream=stream)
            moe.moe_ffn_grouped(x, self.ids, self.w, w13, w2, sfa13, sfa2, self.aligned, self.b, y=self.y,
                                ws=self.ws, stream=stream)
        else:
            moe.moe_ffn_decode(x, self.ids, self.w, w13, w2, y=self.y, ws=self.ws, stream=stream)

    def launch_layer(self, i: int, stream):
        """The layer call of step i alone, on that input's routing computed
        ahead of time (one kernel at one token: routing included)."""
        moe, wl = self.moe, self.wl
        j, (w13, w2, (sfa13, sfa2)) = i % self.n_inputs, self.layers[i % self.L]
        if self.routed_in_layer:
            self.launch_step(i, stream)
            return
        if self.path == "grouped":
            al = self.aligned_all[0 if self.awq else j]
            moe.moe_ffn_grouped(self.x_all[j], self.ids_all[j], self.w_all[j], w13, w2, sfa13, sfa2, al, self.b,
                                y=self.y, ws=self.ws, stream=stream)
        else:
            moe.moe_ffn_decode(self.x_all[j], self.ids_all[j], self.w_all[j], w13, w2, y=self.y, ws=self.ws,
                               stream=stream)

    def graph(self, i0: int, n: int, layer_only: bool = False):
        """A CUDA graph of steps i0 .. i0+n-1 back to back on self.stream."""
        fn = self.launch_layer if layer_only else self.launch_step
        with torch.cuda.stream(self.stream):
            fn(i0, self.stream)                  # warm (outside capture)
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(i0, i0 + n):
                fn(i, self.stream)
        self.stream.synchronize()
        return g

    def bytes_of(self, i0: int, n: int, layer_only: bool = False) -> float:
        f = layer_bytes if (layer_only and not self.routed_in_layer) else step_bytes
        return float(sum(f(self.wl, self.step_ids(i), self.path) for i in range(i0, i0 + n)))

    # ---- descriptions
    def layer_kernels(self) -> str:
        if self.awq and self.path == "grouped":
            return "moe_ffn_grouped (AWQ-4bit): ga::gather + ga::gemm_kernel (both GEMMs, one persistent kernel) + combine"
        if self.nv4 and self.path == "grouped":
            return ("moe_ffn_grouped (NVFP4S, W4A4): ga::gather_nv4_kernel (Q_a of x) + ga::gemm_kernel<Nv4> "
                    "(both GEMMs, weights expanded on chip, Q_a of h in the epilogue) + combine")
        if self.nv4 and self.routed_in_layer:
            return ("moe_ffn_decode_logits (NVFP4S): dpn::pipe_kernel (top-k routing + gate/up + SwiGLU + down + "
                    "routing-weighted sum), one kernel")
        if self.nv4:
            return "moe_ffn_decode (NVFP4S): dn4::gate_up_kernel + dn4::down_kernel"
        if self.awq_pipe:
            return "moe_ffn_decode (AWQ-4bit): dpa::pipe_kernel (gate/up + SwiGLU + down + weighted sum), one kernel"
        if self.awq:
            return "moe_ffn_decode (AWQ-4bit): decode_gate_up_kernel<AWQ> + decode_down_kernel<AWQ>"
        if self.path == "grouped":
            return "moe_ffn_grouped: act_quant + gemm_kernel (both GEMMs, one persistent kernel) + combine"
        if self.routed_in_layer:
            return ("moe_ffn_decode_logits: dp::pipe_kernel (top-k routing + gate/up + SwiGLU + down + "
                    "routing-weighted sum), one kernel")
        return "moe_ffn_decode: ds::gate_up_kernel + ds::down_kernel, PDL-chained"

    def path_text(self) -> str:
        wl = self.wl
        if self.awq and self.path == "grouped":
            return ("expert-centric grouped AWQ (align + gather + tcgen05 kind::f16 GEMM1/GEMM2 on weights "
                    "dequantized in shared memory + combine, b=%d), fixed routing" % self.b)
        if self.nv4 and self.path == "grouped":
            return ("expert-centric grouped NVFP4S W4A4 (topk + align + Q_a gather + tcgen05 kind::f16 GEMM1/GEMM2 "
                    "on weights expanded in tensor memory + combine, b=%d)" % self.b)
        if self.nv4 and self.routed_in_layer:
            return ("single-token NVFP4S decode: routing + gate/up + SwiGLU + down in one kernel, h exchanged "
                    "through L2, activations kept exact")
        if self.nv4:
            return "output-centric NVFP4S decode (topk + gate/up + down, activations kept exact)"
        if self.awq_pipe:
            return ("single-token AWQ decode: gate/up + SwiGLU + down in one kernel, h exchanged through L2, "
                    "fixed routing")
        if self.awq:
            return "output-centric AWQ decode (gate/up + down on CUDA cores), fixed routing"
        if self.path == "grouped":
            return "expert-centric grouped (topk + align + act-quant + tcgen05 GEMM1/GEMM2 + combine, b=%d)" % self.b
        if self.routed_in_layer:
            return "single-token decode: routing + gate/up + SwiGLU + down in one kernel, h exchanged through L2"
        return "output-centric decode (topk + gate/up + down)"

    def launches_per_step(self) -> int:
        if self.path == "grouped":
            na = 2 if self.ws_align is not None else 1
            # (top-k), alignment, act-quant or gather, the GEMM kernel, combine
            return (0 if self.awq else 1) + na + 3
        if self.awq:
            return 1 if self.awq_pipe else 2
        return 1 if self.routed_in_layer else 3


def host_topk_ids(logits: np.ndarray, k: int) -> np.ndarray:
    """Top-k expert ids by logit (stable sort: ties to the lower id), used
    only to count the distinct experts a step touches for the byte count."""
    return np.argsort(-logits, axis=1, kind="stable")[:, :k]


def roofline_obj(st, wl, total_ms, K, total_bytes, world):
    """Roofline of the layer call (the dominant kernels of the step), timed
    alone with CUDA events on its stream: total_ms over K calls moving
    total_bytes of algorithmic traffic.  HBM-bound unless the layer's FLOPs
    at the MXFP8 tensor peak take longer than its bytes at the HBM peak."""
    peak_gbs, peak_kind = measured_peak()
    peak_tf, tf_kind = measured_mxfp8_tflops()
    sec = total_ms * 1e-3
    flops = 2.0 * wl.M * wl.k * 3 * wl.I * wl.d * K * world
    t_hbm = total_bytes / (peak_gbs * 1e9)
    t_mma = flops / (peak_tf * 1e12)
    kern = st.layer_kernels()
    src = (("awq" if st.path == "grouped" else "awq_decode") if st.awq else
           ("nv4" if st.path == "grouped" else "nv4_decode") if st.nv4 else st.path)
    key = f"{st.path}:{wl.name}"
    traffic = committed_traffic(key, decode_src_hash(src))
    if t_mma > t_hbm:
        ach = flops / sec / 1e12 / world
        return {"kernel": kern, "bound": "tensor", "achieved": round(ach, 1), "peak": peak_tf,
                "peak_kind": tf_kind, "unit": "TFLOP/s", "frac": round(ach / peak_tf, 4), "traffic": traffic,
                "us_per_launch": round(total_ms * 1e3 / K, 3),
                "algorithmic_flops_per_launch": round(flops / K / world),
                "hbm_frac": round(total_bytes / sec / 1e9 / world / peak_gbs, 4)}
    ach = total_bytes / sec / 1e9 / world
    return {"kernel": kern, "bound": "hbm", "achieved": round(ach, 1), "peak": peak_gbs, "peak_kind": peak_kind,
            "unit": "GB/s", "frac": round(ach / peak_gbs, 4), "traffic": traffic,
            "us_per_launch": round(total_ms * 1e3 / K, 3),
            "algorithmic_bytes_per_launch": round(total_bytes / K / world),
            "tensor_frac": round(flops / sec / 1e12 / world / peak_tf, 4)}


def gather_replicas(times, sizes, world, device=None):
    """Whole-job figures of N independent replicas: the slowest rank's time
    (MAX over ranks) for each entry of `times` and the SUM over ranks of each
    entry of `sizes`.  Every rank gets the result; world == 1 returns the
    inputs unchanged."""
    times, sizes = [float(v) for v in times], [float(v) for v in sizes]
    if world <= 1:
        return times, sizes
    tmax = torch.tensor(times, dtype=torch.float64, device=device)
    tsum = torch.tensor(sizes, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(tmax, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(tsum, op=torch.distributed.ReduceOp.SUM)
    return tmax.tolist(), tsum.tolist()


def read_flush(buf):
    """Evict the L2 by reading a buffer several times its size: a read leaves
    no dirty lines behind, so nothing is written back during the next step."""
    torch.sum(buf, dim=0, keepdim=True)


def run_ours(args, rank, world, device):
    wl = workload_from_name(args.workload)
    K, W = args.steps, args.warmup
    path, block = args.path, args.block
    if path == "auto":
        # the library's choice at the measured crossover of the two paths
        import top_moe_expert_gb300 as moe
        fmt = {"awq4": moe.MOE_W_AWQ4, "nvfp4s": moe.MOE_W_NVFP4S}.get(wl.fmt, moe.MOE_W_MXFP8)
        p, b = moe.moe_ffn_select_path(wl.M, wl.k, wl.E, wl.d, wl.I, fmt)
        path = "decode" if p == moe.MOE_PATH_DECODE else "grouped"
        block = block or b
    Kg = min(K, 1000 if wl.M <= 64 else 50)              # steps per captured graph
    n_inputs = min(Kg + W, 1024 if wl.M <= 64 else 16)
    st = Step(wl, n_inputs, device, path, block, args.layers)
    s = st.stream

    # ---- the timed steps: graphs of Kg steps back to back (inputs already in
    # HBM, each step on its own input and the next layer copy: no L2 flush)
    R, rem = divmod(K, Kg)
    g_main = st.graph(0, Kg)
    g_rem = st.graph(0, rem) if rem else None
    g_warm = st.graph(0, W)
    steps_bytes = R * st.bytes_of(0, Kg) + (st.bytes_of(0, rem) if rem else 0.0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    torch.cuda.synchronize()
    g_warm.replay()
    torch.cuda.synchronize()
    sampler.start()
    t_keep = time.perf_counter()
    while time.perf_counter() - t_keep < 0.25:         # the sampler sees the GPU busy before the timed region
        g_main.replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(s):
        ev0.record(s)
        for _ in range(R):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t_wall0, t_wall1)
    total_ms = ev0.elapsed_time(ev1)
    del g_rem, g_warm

    # ---- the layer call alone, back to back (routing computed ahead of time
    # for each input): the roofline of the dominant kernel(s)
    Kl = min(K, Kg)
    g_layer = st.graph(0, Kl, layer_only=True)
    Rl = max(1, min(R, 20))
    layer_bytes_total = Rl * st.bytes_of(0, Kl, layer_only=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ev0.record(s)
        for _ in range(Rl):
            g_layer.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    layer_ms = ev0.elapsed_time(ev1)
    del g_layer

    # ---- one isolated call (a one-step graph), L2 evicted by a read before it
    Kc = min(K, 300)
    flushbuf = torch.ones(2 ** 28, dtype=torch.float32, device=device)      # 1 GiB
    g_one = st.graph(0, 1)
    c0 = [torch.cuda.Event(enable_timing=True) for _ in range(Kc)]
    c1 = [torch.cuda.Event(enable_timing=True) for _ in range(Kc)]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(Kc):
            read_flush(flushbuf)
            c0[i].record(s)
            g_one.replay()
            c1[i].record(s)
    torch.cuda.synchronize()
    call_us = sorted(a.elapsed_time(b) * 1e3 for a, b in zip(c0, c1))
    call_bytes = st.bytes_of(0, 1)
    del g_one

    del flushbuf

    # ---- e2e: the same steps through the public API with host buffers
    # (pinned): every step's inputs copied in and its y copied out inside the
    # timed interval; Ke steps back to back in one CUDA graph, as the timed
    # steps are (each on its own input and the next layer copy, no L2 flush),
    # one pair of CUDA events around the replay
    Ke = min(K, 1000)
    rows = list(range(min(Ke, st.n_inputs)))
    io_pin = torch.cat([getattr(st, n)[rows].reshape(len(rows), -1).view(torch.uint8) for n in st.io_host],
                       dim=1).pin_memory()
    assert io_pin.shape[1] == st.io.numel()
    y_pin = torch.empty((Ke, wl.M, wl.d), dtype=torch.bfloat16).pin_memory()

    def e2e_step(i):
        st.io.copy_(io_pin[i % len(rows)], non_blocking=True)
        st.launch_step(i % len(rows), s, x=st.x, logits=st.logits)
        y_pin[i].copy_(st.y, non_blocking=True)

    with torch.cuda.stream(s):
        e2e_step(0)                              # warm (outside capture)
    s.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=s):
        for i in range(Ke):
            e2e_step(i)
    s.synchronize()
    with torch.cuda.stream(s):
        g_e2e.replay()                           # warm replay
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ev0.record(s)
        g_e2e.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    e2e_ms = ev0.elapsed_time(ev1)
    del g_e2e
    e2e_bytes = st.bytes_of(0, Ke) if Ke <= st.n_inputs else float(
        sum(step_bytes(wl, st.step_ids(i % len(rows)), st.path) for i in range(Ke)))

    (total_ms, e2e_ms, layer_ms), (steps_bytes, e2e_bytes, layer_bytes_total) = gather_replicas(
        [total_ms, e2e_ms, layer_ms], [steps_bytes, e2e_bytes, layer_bytes_total], world, device)
    if rank != 0:
        return None

    tbps = steps_bytes / (total_ms * 1e-3) / 1e12
    us_step = total_ms * 1e3 / K
    med_call = call_us[len(call_us) // 2]
    line = {
        "metric": METRIC,
        "value": round(tbps, 4),
        "unit": "TB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(total_ms / K, 6),
        "us_per_layer": round(us_step, 3),
        "tokens_per_s": round(wl.M * world / (total_ms * 1e-3 / K), 1),
        "frac_of_8TBps": round(tbps / world / 8.0, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("awq4-weights/fp16-act/f32-accum" if st.awq else
                  ("nvfp4s-weights/nvfp4-act/f32-accum" if st.path == "grouped" else
                   "nvfp4s-weights/bf16-act/f32-accum") if st.nv4 else "mxfp8-weights/bf16-act/f32-accum"),
        "data": ("synthetic (seeded uniform 4-bit q and zeros, fp16 group scales U(0.005, 0.02), N(0,1) fp16 "
                 "activations, the fixture-A routing of the packed-AWQ study)" if st.awq else
                 ("synthetic (seeded random admissible paired 4:8 NVFP4 packing: uniform E2M1 codes and "
                  "patterns, UE4M3 scales in [0.5, 2], alpha 0.01; N(0,1) bf16 activations; N(0,1) router "
                  "logits, fresh routing every step%s)" % (
                      f"; activation scales alpha_x {st.alpha_x:.3e}, alpha_h {st.alpha_h:.3e}"
                      if st.alpha_x else "")) if st.nv4 else
                 "synthetic (seeded N(0,0.02) weights quantized to MXFP8, N(0,1) bf16 activations, "
                 "N(0,1) router logits; fresh routing every step)"),
        "config": {"workload": wl.name, "M": wl.M, "d": wl.d, "I": wl.I, "E": wl.E, "k": wl.k,
                   "path": st.path_text() + ", CUDA graphs",
                   "l2": (f"not flushed: inputs larger than L2 -- each step reads the next of {st.L} copies of the "
                          f"layer's weights ({st.L * st.layer_weight_bytes / 1e9:.1f} GB, a model's stack of MoE "
                          f"layers) with its own fresh input, so its weights were last read "
                          f"{st.L} steps earlier"),
                   "timing": (f"{K} steps back to back in CUDA graphs of {Kg} steps, one pair of CUDA events "
                              f"around all of them"),
                   "parallelism": f"replicas x{world}"},
        "latency_us": {"median": round(med_call, 3), "p10": round(call_us[len(call_us) // 10], 3),
                       "p90": round(call_us[len(call_us) * 9 // 10], 3), "calls": Kc,
                       "tbps_at_median": round(call_bytes / (med_call * 1e-6) / 1e12, 4),
                       "how": "one step alone (a one-step graph between CUDA events), the L2 evicted by a "
                              "1 GiB read before each call"},
        "e2e": {"value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TB/s",
                "us_per_layer": round(e2e_ms * 1e3 / Ke, 3), "steps": Ke,
                "h2d_bytes_per_step": st.io.numel(),
                "d2h_bytes_per_step": wl.M * wl.d * 2,
                "how": (f"{Ke} steps back to back in one CUDA graph, each: the copy of its x and logits from "
                        "pinned host memory, the library call, the copy of y to pinned host memory; one pair of "
                        "CUDA events around the replay")},
        "gpu_launches": st.launches_per_step() * K,
        "roofline": roofline_obj(st, wl, layer_ms, Rl * Kl, layer_bytes_total, world),
        "clocks": clocks,
        "wall_s_timed_loop": round(t_wall1 - t_wall0, 3),
        "_path": st.path,
    }
    return line


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def cpu_baseline(wl, device, path="decode", seconds=8.0):
    """The oracle, as it stands, on the host cores: single-thread (one
    token per call) and all-core (one token per core per call, each token a
    step of its own with fresh routing; the oracle parallelises over tokens),
    until ~`seconds` of timed CPU work each.  The oracle runs in the mode the
    path computes (exact for decode, block-scaled for grouped).  Expert weights
    are quantized by the oracle from the same fp32 draws (set-up, not timed)."""
    import oracle
    from top_moe_expert_gb300 import inputs
    if wl.fmt == "awq4":
        return _cpu_baseline_awq(wl, seconds)
    if wl.fmt == "nvfp4s":
        return _cpu_baseline_nv4(wl, path, seconds)
    cache = {}

    def expert(which, e):
        if (which, e) not in cache:
            f = inputs.weights_fp32_device(wl, which, e, device).cpu().numpy().astype(np.float64)
            cache[(which, e)] = oracle.mxfp8_quantize(f)
        return cache[(which, e)]

    mode = oracle.MODE_MX if path == "grouped" else oracle.MODE_EXACT
    ncores = os.cpu_count() or 1

    def run(threads, S):
        oracle.set_num_threads(threads)
        t_total, nbytes, calls, seed = 0.0, 0, 0, 10_000
        while t_total < seconds and calls < 64:
            # S tokens, each with the routing and activation of a step of its own
            logits = np.concatenate([inputs.router_logits(wl, seed + t)[:1] for t in range(S)])
            x = torch.cat([inputs.activations(wl, seed + t)[:1] for t in range(S)]).to(torch.float64).numpy()
            ids, _ = oracle.topk_softmax(logits, wl.k)
            experts = sorted(set(ids.reshape(-1).tolist()))
            slot = np.full(wl.E, -1, dtype=np.int32)
            slot[experts] = np.arange(len(experts), dtype=np.int32)
            ws = {}
            for which in ("w13", "w2"):
                qs = [expert(which, e) for e in experts]
                ws[which] = {"fmt": "mxfp8", "q": np.stack([q for q, _ in qs]),
                             "s": np.stack([s for _, s in qs]), "slot": slot}
            t0 = time.perf_counter()
            ids2, w2 = oracle.topk_softmax(logits, wl.k)
            oracle.moe_layer(x, ids2, w2, wl.E, ws["w13"], ws["w2"], mode=mode)
            t_total += time.perf_counter() - t0
            # each token is one step of the M=1 workload: its own distinct experts
            nbytes += sum(len(np.unique(ids[t])) * expert_bytes(wl) + 4 * wl.d + 4 * wl.E for t in range(S))
            calls += 1
            seed += S
        return nbytes / t_total / 1e12, calls, t_total

    v1, c1, t1 = run(1, 1)
    vn, cn, tn = run(ncores, ncores)
    oracle.set_num_threads(ncores)
    return {"value": vn, "unit": "TB/s", "cores": ncores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": (f"{cn} calls of {ncores} tokens (each token one step of {wl.name}: top-k + layer, binary64, "
                       f"{'block-scaled' if mode else 'exact'} mode, its own fresh routing), {ncores} OpenMP "
                       f"threads, {tn:.1f} s timed"),
            "single_thread": {"value": v1, "unit": "TB/s", "cores": 1,
                              "sample": f"{c1} single-token steps, 1 thread, {t1:.1f} s timed",
                              "us_per_token": round(t1 / c1 * 1e6, 1)},
            "us_per_token": round(tn / (cn * ncores) * 1e6, 1)}


def _cpu_baseline_awq(wl, seconds):
    """The oracle on the AWQ layer (fp16 h, as the grouped path computes):
    the fixed routing of the first 4 tokens per step."""
    import oracle
    from top_moe_expert_gb300 import inputs
    S = min(wl.M, 4)
    ids = inputs.fixture_a_ids(wl.M, wl.k, wl.E)[:S]
    w = inputs.fixture_a_weights(wl.M, wl.k, wl.seed)[:S].astype(np.float64)
    experts = sorted(set(ids.reshape(-1).tolist()))
    slot = np.full(wl.E, -1, dtype=np.int32)
    slot[experts] = np.arange(len(experts), dtype=np.int32)
    ws = {}
    for which in ("w13", "w2"):
        q, sc, z = inputs.awq_weights(wl, which, experts)
        ws[which] = {"fmt": "awq4", "q": q, "s": sc, "z": z, "slot": slot}
    t_total, nbytes, steps = 0.0, 0, 0
    while t_total < seconds and steps < 64:
        x = inputs.activations(wl, 10_000 + steps, dtype=torch.float16)[:S].to(torch.float64).numpy()
        t0 = time.perf_counter()
        oracle.moe_layer(x, ids, w, wl.E, ws["w13"], ws["w2"], mode=oracle.MODE_H16)
        t_total += time.perf_counter() - t0
        nbytes += len(experts) * expert_bytes(wl) + S * 4 * wl.d
        steps += 1
    threads = min(oracle.num_threads(), S)
    return {"value": nbytes / t_total / 1e12, "unit": "TB/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} steps (layer, binary64, fp16-h mode) of {wl.name} on {S} token(s) each, "
                      f"fixed routing, {t_total:.1f} s timed",
            "us_per_token": round(t_total / steps / S * 1e6, 1)}


def _nv4_sample(wl, path, seed, S):
    """S tokens of the NVFP4S workload, each with its own routing, and the
    packed weights of the experts they touch (oracle format dicts)."""
    import oracle
    from top_moe_expert_gb300 import inputs
    logits = np.concatenate([inputs.router_logits(wl, seed + t)[:1] for t in range(S)])
    x = torch.cat([inputs.activations(wl, seed + t)[:1] for t in range(S)]).to(torch.float64).numpy()
    ids, w = oracle.topk_softmax(logits, wl.k)
    experts = sorted(set(ids.reshape(-1).tolist()))
    slot = np.full(wl.E, -1, dtype=np.int32)
    slot[experts] = np.arange(len(experts), dtype=np.int32)
    ws = {}
    for which in ("w13", "w2"):
        v, m, sc, a = inputs.nvfp4s_weights(wl, which, experts)
        ws[which] = {"fmt": "nvfp4s", "v": v, "m": m, "s": sc, "alpha": a, "slot": slot}
    return logits, x, ids, w, ws


def _cpu_baseline_nv4(wl, path, seconds):
    """The oracle on the NVFP4S layer: exact activations (decode path) or
    the W4A4 mode (grouped path), S tokens per call, each with its own
    routing; all cores."""
    import oracle
    S = os.cpu_count() or 1
    a_x, a_h = 5.0 / (6 * 448), 16.0 / (6 * 448)
    t_total, nbytes, calls, seed = 0.0, 0, 0, 10_000
    while t_total < seconds and calls < 64:
        logits, x, ids, _, ws = _nv4_sample(wl, path, seed, S)
        t0 = time.perf_counter()
        ids2, w2 = oracle.topk_softmax(logits, wl.k)
        if path == "grouped":
            oracle.moe_layer_a4(x, ids2, w2, wl.E, ws["w13"], ws["w2"], a_x, a_h)
        else:
            oracle.moe_layer(x, ids2, w2, wl.E, ws["w13"], ws["w2"])
        t_total += time.perf_counter() - t0
        nbytes += sum(len(np.unique(ids[t])) * expert_bytes(wl, path) + 4 * wl.d + 4 * wl.E for t in range(S))
        calls += 1
        seed += S
    return {"value": nbytes / t_total / 1e12, "unit": "TB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": (f"{calls} calls of {S} tokens (each token one step of {wl.name}: top-k + layer, binary64, "
                       f"{'W4A4' if path == 'grouped' else 'exact-activation'} mode, its own routing), "
                       f"{t_total:.1f} s timed"),
            "us_per_token": round(t_total / (calls * S) * 1e6, 1)}


def _reference_awq(args, wl, world):
    """--impl reference on the AWQ layer: each step one routed expert of
    token 0 restricted to its first 128 neurons (one AWQ group of the down
    projection), binary64 with fp16 h."""
    import oracle
    from top_moe_expert_gb300 import inputs
    K, W = args.steps, args.warmup
    Is = 128
    e0 = int(inputs.fixture_a_ids(wl.M, wl.k, wl.E)[0, 0])
    q13, s13, z13 = inputs.awq_weights(wl, "w13", [e0])
    q2, s2, z2 = inputs.awq_weights(wl, "w2", [e0])
    I = wl.I
    rows = np.r_[0:Is, I:I + Is]
    zrows = np.r_[0:Is // 8, I // 8:I // 8 + Is // 8]
    slot = np.full(wl.E, -1, dtype=np.int32)
    slot[e0] = 0
    w13 = {"fmt": "awq4", "q": q13[:, rows], "s": s13[:, rows], "z": z13[:, zrows], "slot": slot}
    kq = Is // 8
    w2 = {"fmt": "awq4", "q": np.ascontiguousarray(q2[:, :, :kq]), "s": np.ascontiguousarray(s2[:, :, :Is // 128]),
          "z": np.ascontiguousarray(z2[:, :, :Is // 128]), "slot": slot}
    x = inputs.activations(wl, 0, dtype=torch.float16).to(torch.float64).numpy()[:1]
    one = np.array([[e0]], dtype=np.int32)
    wone = np.ones((1, 1))
    per = 3 * Is * wl.d
    sample_bytes = per // 2 + per // 128 * 2 + per // 256 + wl.d * 2 + wl.d * 2
    nbytes, t_total = 0, 0.0
    for i in range(W + K):
        t0 = time.perf_counter()
        oracle.moe_layer(x, one, wone, wl.E, w13, w2, mode=oracle.MODE_H16)
        dt = time.perf_counter() - t0
        if i >= W:
            t_total += dt
            nbytes += sample_bytes
    v = nbytes / t_total / 1e12
    sample = (f"one routed expert of one token, first {Is} intermediate neurons, binary64 with fp16 h, "
              f"{oracle.num_threads()} OpenMP thread(s) available (one token: 1 used)")
    return {"metric": METRIC, "impl": "reference", "value": v, "unit": "TB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": t_total * 1e3 / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "M": wl.M, "d": wl.d, "I": wl.I, "E": wl.E, "k": wl.k,
                       "path": "CPU oracle (sample)"},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": sample, "value": v, "unit": "TB/s"},
            "e2e": {"value": v, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def _reference_nv4(args, wl, world):
    """--impl reference on the NVFP4S layer: each step one token (its own
    routing, all k experts) through the oracle in the path's mode, 1 thread."""
    import oracle
    K, W = args.steps, args.warmup
    path = "grouped" if args.path == "grouped" else "decode"
    oracle.set_num_threads(1)
    a_x, a_h = 5.0 / (6 * 448), 16.0 / (6 * 448)
    nbytes, t_total = 0, 0.0
    for i in range(W + K):
        logits, x, ids, w, ws = _nv4_sample(wl, path, 20_000 + i, 1)
        t0 = time.perf_counter()
        if path == "grouped":
            oracle.moe_layer_a4(x, ids, w, wl.E, ws["w13"], ws["w2"], a_x, a_h)
        else:
            oracle.moe_layer(x, ids, w, wl.E, ws["w13"], ws["w2"])
        dt = time.perf_counter() - t0
        if i >= W:
            t_total += dt
            nbytes += len(np.unique(ids)) * expert_bytes(wl, path) + 4 * wl.d
    v = nbytes / t_total / 1e12
    sample = f"per step: one token of {wl.name} (all its routed experts), binary64 oracle, 1 thread"
    return {"metric": METRIC, "impl": "reference", "value": v, "unit": "TB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": t_total * 1e3 / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "M": wl.M, "d": wl.d, "I": wl.I, "E": wl.E, "k": wl.k,
                       "path": "CPU oracle (sample)"},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "sample": sample, "value": v, "unit": "TB/s"},
            "e2e": {"value": v, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    import oracle
    from top_moe_expert_gb300 import inputs
    wl = workload_from_name(args.workload)
    oracle.build()
    device = torch.device("cuda", 0) if torch.cuda.is_available() else None
    # Each step is a bounded sample of the workload: one routed expert of one
    # token restricted to its first 64 intermediate neurons (gate/up rows
    # 0..63, down columns 0..63), so K+W steps stay within a few minutes.
    K, W = args.steps, args.warmup
    if wl.fmt == "awq4":
        return _reference_awq(args, wl, world)
    if wl.fmt == "nvfp4s":
        return _reference_nv4(args, wl, world)
    Is = 64
    logits = inputs.router_logits(wl, 0)
    ids, _ = oracle.topk_softmax(logits, wl.k)
    e0 = int(ids[0, 0])
    def draw(which):
        if device is not None:
            return inputs.weights_fp32_device(wl, which, e0, device).cpu().numpy()
        return inputs.weights_fp32(wl, which, [e0])[0]
    f13 = draw("w13")
    f13 = np.concatenate([f13[:Is], f13[wl.I:wl.I + Is]])[None].astype(np.float64)
    f2 = draw("w2")[:, :Is][None].astype(np.float64)
    slot = np.full(wl.E, -1, dtype=np.int32)
    slot[e0] = 0
    q13, s13 = oracle.mxfp8_quantize_3d(f13)
    q2, s2 = oracle.mxfp8_quantize_3d(f2)
    w13 = {"fmt": "mxfp8", "q": q13, "s": s13, "slot": slot}
    w2 = {"fmt": "mxfp8", "q": q2, "s": s2, "slot": slot}
    x = inputs.activations(wl, 0).to(torch.float64).numpy()[:1]
    one = np.array([[e0]], dtype=np.int32)
    wone = np.ones((1, 1))
    sample_bytes = 3 * Is * wl.d * 33 // 32 + wl.d * 2 + wl.d * 2
    nbytes, t_total = 0, 0.0
    for i in range(W + K):
        t0 = time.perf_counter()
        oracle.moe_layer(x, one, wone, wl.E, w13, w2)
        dt = time.perf_counter() - t0
        if i >= W:
            t_total += dt
            nbytes += sample_bytes
    v = nbytes / t_total / 1e12
    return {"metric": METRIC, "impl": "reference", "value": v, "unit": "TB/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": t_total * 1e3 / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "M": wl.M, "d": wl.d, "I": wl.I, "E": wl.E, "k": wl.k},
            "cpu_baseline": {"value": v, "unit": "TB/s", "cores": 1, "kind": "oracle",
                             "sample": f"per step: one routed expert of one token of {wl.name}, "
                                       f"first {Is} intermediate neurons (binary64 oracle, 1 thread)"},
            "e2e": {"value": v, "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------ Table 8 sweep

TABLE8 = {
    # model: (d, I, N sweep, G sweep) -- gate/up (2I, d) and down (d, I) of the
    # grouped-GEMM benchmark shapes ("Hardware-Native Joint Sparse-
    # Quantization ...", App. D.2, Table 8)
    "qwen": (2048, 768, (16, 32, 64, 128, 256, 512, 1024), (8, 16, 32, 64, 128)),
    "kimi": (7168, 2048, (32, 64, 128, 256, 512, 1024), (24, 48, 96, 192, 384)),
}


def run_table8(model: str, device, reps: int = 20, out=sys.stdout, fmt: str = "mxfp8"):
    """The grouped layer over the benchmark's (N, G) grid with per-expert token
    counts {N, 3N/4, N/2, N/4} repeated over the G experts (one route per
    token, weight 1), on the aligned and on the fixed-capacity layout.  One
    step is the alignment and the layer call (activation quantization, both
    GEMMs, combine), timed back to back in a CUDA graph over copies of the
    weights that together exceed the L2.  One JSON line per (G, N, layout):
    the page's effective TFLOP/s (2 * (2I*d + d*I) * sum N_g / t) and the
    fraction of the measured HBM bandwidth the weight and activation bytes
    reach.  fmt "nvfp4s": the paired 4:8 sparse NVFP4 W4A4 grouped path (the
    page's own format) on random admissible packing, aligned layout only."""
    import top_moe_expert_gb300 as moe
    from top_moe_expert_gb300 import inputs
    d, I, Ns, Gs = TABLE8[model]
    peak_gbs, _ = measured_peak()
    nv4 = fmt == "nvfp4s"
    for G in Gs:
        wl = inputs.Workload(f"table8_{model}_g{G}", M=1, d=d, I=I, E=G, k=1, seed=30)
        # weight bytes: NVFP4S kept codes and side records (3/8 byte a weight) and two factors per expert
        lw = G * 3 * I * d * 3 // 8 + 8 * G if nv4 else G * 3 * I * d * 33 // 32
        n_copies = max(1, min(8, -(-4 * 130 * 2 ** 20 // lw)))
        layers = []
        # NVFP4S activation scales, constants of the layer: N(0,1) inputs up to 6.5,
        # |h| up to 16 (the weights' RMS gives |g|, |u| of order 1)
        a_x, a_h = 6.5 / (6 * 448), 16.0 / (6 * 448)
        for c in range(n_copies):
            if nv4:
                v13, m13, c13, al13 = inputs.nvfp4s_weights_device(wl, "w13", device)
                v2, m2, c2, al2 = inputs.nvfp4s_weights_device(wl, "w2", device)
                w13 = moe.Weights(moe.MOE_W_NVFP4S, v13, c13, m13, al13)
                w2 = moe.Weights(moe.MOE_W_NVFP4S, v2, c2, m2, al2)
                layers.append((w13, w2, moe.moe_grouped_prepare_nvfp4s(w13, w2, a_x, a_h)))
                continue
            q13 = torch.empty((G, 2 * I, d), dtype=torch.uint8, device=device)
            s13 = torch.empty((G, 2 * I, d // 32), dtype=torch.uint8, device=device)
            q2 = torch.empty((G, d, I), dtype=torch.uint8, device=device)
            s2 = torch.empty((G, d, I // 32), dtype=torch.uint8, device=device)
            for e in range(G):
                if c == 0:
                    moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w13", e, device), q13[e], s13[e])
                    moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w2", e, device), q2[e], s2[e])
            if c > 0:
                q13.copy_(layers[0][0].q); s13.copy_(layers[0][0].scale)
                q2.copy_(layers[0][1].q); s2.copy_(layers[0][1].scale)
            w13, w2 = moe.Weights(moe.MOE_W_MXFP8, q13, s13), moe.Weights(moe.MOE_W_MXFP8, q2, s2)
            layers.append((w13, w2, moe.moe_grouped_prepare(w13, w2)))
        for N in Ns:
            ids_np = inputs.imbalanced_routing(N, G)
            M = ids_np.shape[0]
            ids = torch.from_numpy(ids_np).to(device)
            w = torch.ones((M, 1), dtype=torch.float32, device=device)
            x = inputs.activations(inputs.Workload("t8x", M=M, d=d, I=I, E=G, k=1, seed=31)).to(device)
            y = torch.empty((M, d), dtype=torch.bfloat16, device=device)
            b = moe.moe_ffn_select_path(M, 1, G, d, I, moe.MOE_W_NVFP4S if nv4 else moe.MOE_W_MXFP8)[1] or 16
            C = -(-N // b) * b
            cr, cb = moe.moe_align_capacity(M, 1, G, b)
            for layout in (("aligned",) if nv4 else ("aligned", "fixed")):
                if layout == "aligned":
                    al = (torch.empty(cr, dtype=torch.int32, device=device),
                          torch.empty(cb, dtype=torch.int32, device=device),
                          torch.empty(1, dtype=torch.int32, device=device))
                    na = moe.moe_align_workspace_size(M, 1, G, b)
                    wsa = torch.empty(max(na, 256), dtype=torch.uint8, device=device) if na else None
                    rows = cr
                else:
                    al = moe.moe_align_fixed_capacity(ids, G, b, C)
                    wsa, rows = None, G * C
                ws = torch.empty(moe.moe_ffn_grouped_workspace_size(M, 1, d, I, b, rows), dtype=torch.uint8,
                                 device=device)
                def step(i):
                    # every launch on the current stream (the capture stream
                    # while the graph is being recorded)
                    w13, w2, sfa = layers[i % n_copies]
                    if layout == "aligned":
                        moe.moe_align_block_size(ids, G, b, out=al, ws=wsa)
                    else:
                        moe.moe_align_fixed_capacity(ids, G, b, C, out=al)
                    moe.moe_ffn_grouped(x, ids, w, w13, w2, sfa[0], sfa[1], al, b, y=y, ws=ws)

                for i in range(3):
                    step(i)
                torch.cuda.synchronize(device)
                n_steps = n_copies * max(1, reps // n_copies)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(n_steps):
                        step(i)
                g.replay()
                torch.cuda.synchronize(device)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(3):
                    g.replay()
                e1.record()
                torch.cuda.synchronize(device)          # the graph is done before its buffers are freed
                us = e0.elapsed_time(e1) * 1e3 / (3 * n_steps)
                flop = 2.0 * (2 * I * d + d * I) * M
                nbytes = lw + M * d * 2 + M * d * 2
                print(json.dumps({"table8": model, "fmt": fmt, "G": G, "N": N, "tokens": M, "layout": layout, "b": b,
                                  "us_per_step": round(us, 2), "eff_tflops": round(flop / (us * 1e-6) / 1e12, 2),
                                  "hbm_frac": round(nbytes / (us * 1e-6) / 1e9 / peak_gbs, 4),
                                  "weight_copies": n_copies}), file=out, flush=True)
                del g, ws, al
                torch.cuda.synchronize(device)
            del ids, w, x, y
        del layers
        torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_m1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "decode", "grouped"])
    ap.add_argument("--block", type=int, default=0, help="MoE block size b of the grouped path (0: automatic)")
    ap.add_argument("--table8", choices=sorted(TABLE8), default=None,
                    help="run the grouped-GEMM benchmark grid (one JSON line per point) instead of the bench line")
    ap.add_argument("--table8-fmt", choices=["mxfp8", "nvfp4s"], default="mxfp8",
                    help="weight format of the --table8 grid (nvfp4s: the W4A4 paired 4:8 sparse path)")
    ap.add_argument("--layers", type=int, default=0,
                    help="copies of the layer's weights the steps rotate through (0: enough that the inputs of "
                         "the timed steps exceed the L2; 1 keeps a profiling run small)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)

    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    import __graft_entry__
    __graft_entry__.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if args.table8:
        run_table8(args.table8, device, fmt=args.table8_fmt)
        return
    line = run_ours(args, rank, world, device)
    if line is not None:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(workload_from_name(args.workload), device, line["_path"])
        line.pop("_path", None)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
