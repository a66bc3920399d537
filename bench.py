#!/usr/bin/env python3
"""Benchmark of the routed MoE expert-FFN layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_m1|tiny|sweep_m<M>[_zipf]|large_m1|large_m8|awq_fixture_a|awq_m1|probe_m16384]

A step is one pass of the hot path over one batch of fresh synthetic input:
top-k routing of the step's router logits, then the layer (output-centric
decode kernels).  The default workload is the 128-expert d=2048 / I=768
top-8 layer at M=1 with MXFP8 weights (623 MB resident), fresh routing every
step.  The L2 is flushed (a 512 MiB write) between timed steps, outside the
timed interval.  Each step's device time is taken with CUDA events on the
launching stream around a CUDA-graph replay of the step.

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
    if name.startswith("sweep_m"):
        rest = name[len("sweep_m"):]
        routing = "zipf" if rest.endswith("_zipf") else "uniform"
        return inputs.sweep(int(rest.split("_")[0]), routing)
    raise SystemExit(f"unknown workload {name}")


def expert_bytes(wl) -> int:
    """Weight bytes of one expert.  MXFP8: 3*I*d codes + 3*I*d/32 scale
    bytes.  AWQ-4bit: 3*I*d/2 packed values + an fp16 scale and a 4-bit zero
    per 128 values."""
    if wl.fmt == "awq4":
        n = 3 * wl.I * wl.d
        return n // 2 + n // 128 * 2 + n // 128 // 2
    return 3 * wl.I * wl.d * 33 // 32


def layer_bytes(wl, ids: np.ndarray) -> int:
    """Algorithmic bytes of one layer call: distinct routed experts' weights,
    x and the routing (ids, weights) read, y written (bf16)."""
    distinct = len(np.unique(ids[(ids >= 0) & (ids < wl.E)]))
    return distinct * expert_bytes(wl) + wl.M * wl.d * 2 + wl.M * wl.k * 8 + wl.M * wl.d * 2


def step_bytes(wl, ids: np.ndarray) -> int:
    """Algorithmic bytes of one step: distinct routed experts' weights, the
    activations read (x, router logits) and the output written (bf16 y)."""
    distinct = len(np.unique(ids[(ids >= 0) & (ids < wl.E)]))
    routing = wl.M * wl.k * 8 if wl.routing == "fixture_a" else wl.M * wl.E * 4   # fixed ids/w, or logits
    return distinct * expert_bytes(wl) + wl.M * wl.d * 2 + routing + wl.M * wl.d * 2


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
                "reasons": sorted(reasons), "samples": len(self.rows)}


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
    "decode": ("decode.cu", "decode_fused.cu", "decode_stream.cu", "decode_m1.cu", "decode_mx_m1.cu",
               "decode_mx_m1.cuh", "decode_awq_m1.cuh", "decode_internal.h", "topk.cu", "topk.cuh", "common.cuh",
               "tc.cuh", "attr.h"),
    "grouped": ("grouped.cu", "grouped_internal.h", "align.cu", "topk.cu", "topk.cuh", "common.cuh", "tc.cuh",
                "attr.h"),
    "awq": ("grouped_awq.cu", "grouped_awq_mma.cu", "grouped_awq_mma.cuh", "decode_awq_m1.cuh", "grouped.cu",
            "grouped_internal.h", "align.cu", "common.cuh", "tc.cuh", "attr.h"),
    "awq_decode": ("decode.cu", "decode_awq_m1.cu", "decode_awq_m1.cuh", "decode_internal.h", "common.cuh",
                   "tc.cuh", "attr.h"),
}


def decode_src_hash(path: str = "decode") -> str:
    """SHA-256 over the kernel sources of one path (the ncu counters in
    profiles/traffic.json are valid only for these exact sources)."""
    h = hashlib.sha256()
    for f in SRC_FILES[path]:
        h.update(open(os.path.join(ROOT, "top_moe_expert_gb300", "csrc", f), "rb").read())
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


class DecodeStep:
    """Device-resident workload + a CUDA graph of one step: top-k routing and
    the layer (decode path), or top-k, alignment and the grouped layer."""

    def __init__(self, wl, nsteps: int, device, path: str = "decode", block: int = 0, w2_layout: str = "auto"):
        import top_moe_expert_gb300 as moe
        from top_moe_expert_gb300 import inputs
        self.moe, self.wl, self.dev, self.path = moe, wl, device, path
        self.routed_in_layer = False
        self.w2_standard = w2_layout == "standard"
        self.awq = wl.fmt == "awq4"
        # the library's opt-in kernels (MOE_FFN_CANDIDATE_KERNELS=1) decide several paths below
        self.cand = bool(moe.moe_candidate_kernels_enabled())
        E, d, I, M, k = wl.E, wl.d, wl.I, wl.M, wl.k
        if self.awq:
            self._init_awq(wl, nsteps, device, block)
            return
        self.q13 = torch.empty((E, 2 * I, d), dtype=torch.uint8, device=device)
        self.s13 = torch.empty((E, 2 * I, d // 32), dtype=torch.uint8, device=device)
        self.q2 = torch.empty((E, d, I), dtype=torch.uint8, device=device)
        self.s2 = torch.empty((E, d, I // 32), dtype=torch.uint8, device=device)
        for e in range(E):
            moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w13", e, device), self.q13[e], self.s13[e])
            moe.moe_mxfp8_quantize(inputs.weights_fp32_device(wl, "w2", e, device), self.q2[e], self.s2[e])
        self.w13 = moe.Weights(moe.MOE_W_MXFP8, self.q13, self.s13)
        self.w2 = moe.Weights(moe.MOE_W_MXFP8, self.q2, self.s2)
        self.fused = False
        if path == "grouped":
            self.b = block or grouped_block(wl)
            self.sfa13, self.sfa2 = moe.moe_grouped_prepare(self.w13, self.w2)
        else:
            # small batches take the single-pass kernel, which reads the down
            # projection neuron-major: pack it once (same bytes, K-outer order)
            self.fused = M <= 4 and d % 1024 == 0 and not self.w2_standard
            # one token on that layout: routing runs inside the layer's kernel
            self.routed_in_layer = self.fused and M == 1 and d in (1024, 2048) and E <= 512
            if self.w2_standard and M == 1 and E <= 512 and self.cand:
                # one token on the standard layout: the single-kernel path, routing inside
                self.routed_in_layer = True
            if self.fused:
                self.w2 = moe.moe_mxfp8_transpose(self.w2)
                del self.q2, self.s2
                torch.cuda.empty_cache()
        # fresh routing and activations for every step (large batches cycle
        # through a pool of distinct steps to bound host memory)
        self.n_inputs = nsteps if M <= 64 else min(nsteps, 16)
        self.logits_host = torch.from_numpy(np.stack([inputs.router_logits(wl, i) for i in range(self.n_inputs)]))
        self.x_host = torch.stack([inputs.activations(wl, i) for i in range(self.n_inputs)])
        self.logits_all = self.logits_host.to(device)
        self.x_all = self.x_host.to(device)
        # x and the router logits share one device buffer, so a step's inputs
        # arrive in one host-to-device copy
        self.io = torch.empty(M * d * 2 + M * E * 4, dtype=torch.uint8, device=device)
        self.x = self.io[:M * d * 2].view(torch.bfloat16).view(M, d)
        self.logits = self.io[M * d * 2:].view(torch.float32).view(M, E)
        self.io_host = ("x_host", "logits_host")     # host tensors packed into io, in order
        self.ids = torch.empty((M, k), dtype=torch.int32, device=device)
        self.w = torch.empty((M, k), dtype=torch.float32, device=device)
        self.y = torch.empty((M, d), dtype=torch.bfloat16, device=device)
        if path == "grouped":
            cr, cb = moe.moe_align_capacity(M, k, E, self.b)
            self.aligned = (torch.empty(cr, dtype=torch.int32, device=device),
                            torch.empty(cb, dtype=torch.int32, device=device),
                            torch.empty(1, dtype=torch.int32, device=device))
            na = moe.moe_align_workspace_size(M, k, E, self.b)
            self.ws_align = torch.empty(max(na, 256), dtype=torch.uint8, device=device) if na else None
            self.ws = torch.empty(moe.moe_ffn_grouped_workspace_size(M, k, d, I, self.b, cr), dtype=torch.uint8,
                                  device=device)
        else:
            self.ws = torch.zeros(moe.moe_ffn_decode_workspace_size(M, k, d, I), dtype=torch.uint8, device=device)
        self.stream = torch.cuda.Stream(device)
        torch.cuda.synchronize()

    def _init_awq(self, wl, nsteps, device, block):
        """The 4-bit AWQ layer on its fixed closed-form routing (fixture A):
        a step is alignment + the grouped layer, or the output-centric decode
        layer alone; activations fp16."""
        moe = self.moe
        from top_moe_expert_gb300 import inputs
        E, d, I, M, k = wl.E, wl.d, wl.I, wl.M, wl.k
        dev_t = lambda a: torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)
        q13, s13, z13 = inputs.awq_weights(wl, "w13")
        q2, s2, z2 = inputs.awq_weights(wl, "w2")
        self.w13 = moe.Weights(moe.MOE_W_AWQ4, dev_t(q13), dev_t(s13).view(torch.float16), dev_t(z13))
        self.w2 = moe.Weights(moe.MOE_W_AWQ4, dev_t(q2), dev_t(s2).view(torch.float16), dev_t(z2))
        del q13, s13, z13, q2, s2, z2
        self.fused = False
        self.b = block or wl.b
        self.sfa13 = self.sfa2 = None
        self.fixed_ids = inputs.fixture_a_ids(M, k, E)
        self.n_inputs = min(nsteps, 64)
        self.logits_host = torch.zeros((self.n_inputs, M, E), dtype=torch.float32)   # routing is fixed
        self.x_host = torch.stack([inputs.activations(wl, i, dtype=torch.float16) for i in range(self.n_inputs)])
        self.logits_all = self.logits_host.to(device)
        self.x_all = self.x_host.to(device)
        self.logits = torch.empty((M, E), dtype=torch.float32, device=device)
        # the routing is fixed: x is the step's only input
        self.io = torch.empty(M * d * 2, dtype=torch.uint8, device=device)
        self.x = self.io.view(torch.float16).view(M, d)
        self.io_host = ("x_host",)
        self.ids = torch.from_numpy(self.fixed_ids).to(device)
        self.w = torch.from_numpy(inputs.fixture_a_weights(M, k, wl.seed)).to(device)
        self.y = torch.empty((M, d), dtype=torch.bfloat16, device=device)
        cr, cb = moe.moe_align_capacity(M, k, E, self.b)
        self.aligned = (torch.empty(cr, dtype=torch.int32, device=device),
                        torch.empty(cb, dtype=torch.int32, device=device),
                        torch.empty(1, dtype=torch.int32, device=device))
        na = moe.moe_align_workspace_size(M, k, E, self.b)
        self.ws_align = torch.empty(max(na, 256), dtype=torch.uint8, device=device) if na else None
        if self.path == "grouped":
            self.ws = torch.empty(moe.moe_ffn_grouped_workspace_size(M, k, d, I, self.b, cr), dtype=torch.uint8,
                                  device=device)
        else:
            self.ws = torch.zeros(moe.moe_ffn_decode_workspace_size(M, k, d, I), dtype=torch.uint8, device=device)
        self.stream = torch.cuda.Stream(device)
        torch.cuda.synchronize()

    def step_ids(self, j: int) -> np.ndarray:
        """Expert ids of input j (to count the distinct experts a step reads)."""
        if self.awq:
            return self.fixed_ids
        return host_topk_ids(self.logits_host[j].numpy(), self.wl.k)

    def launch_pre(self, stream=None):
        """Routing of the step: top-k (and, for the grouped path, alignment);
        nothing when the layer call routes the token itself."""
        moe = self.moe
        if self.routed_in_layer:
            return
        if self.awq:
            if self.path == "grouped":
                moe.moe_align_block_size(self.ids, self.wl.E, self.b, out=self.aligned, ws=self.ws_align,
                                         stream=stream)
            return
        moe.moe_topk_softmax(self.logits, self.wl.k, self.ids, self.w, stream=stream)
        if self.path == "grouped":
            moe.moe_align_block_size(self.ids, self.wl.E, self.b, out=self.aligned, ws=self.ws_align, stream=stream)

    def launch_layer(self, stream=None):
        """The layer call itself (one C-ABI call)."""
        moe = self.moe
        if self.path == "grouped":
            moe.moe_ffn_grouped(self.x, self.ids, self.w, self.w13, self.w2, self.sfa13, self.sfa2, self.aligned,
                                self.b, y=self.y, ws=self.ws, stream=stream)
        elif self.routed_in_layer:
            moe.moe_ffn_decode_logits(self.logits, self.x, self.wl.k, self.w13, self.w2, y=self.y, topk_ids=self.ids,
                                      topk_w=self.w, ws=self.ws, stream=stream)
        else:
            moe.moe_ffn_decode(self.x, self.ids, self.w, self.w13, self.w2, y=self.y, ws=self.ws, stream=stream)

    def launch(self, stream=None):
        self.launch_pre(stream)
        self.launch_layer(stream)

    def layer_kernels(self) -> str:
        if self.awq and self.path == "grouped" and self.b <= 16 and self.cand:
            return ("moe_ffn_grouped (AWQ-4bit, b <= 16): gsm::awq_mma_kernel (both GEMMs on mma.sync over the raw "
                    "codes, one kernel) + combine")
        if self.awq and self.path == "grouped":
            return "moe_ffn_grouped (AWQ-4bit): ga::gather + ga::gemm_kernel (both GEMMs, one persistent kernel) + combine"
        if self.awq and self.wl.M == 1 and self.cand:
            return "moe_ffn_decode (AWQ-4bit, one token): da1::awq_m1_kernel (gate/up + SwiGLU + down), one kernel"
        if self.awq and 2 <= self.wl.M <= 64 and self.cand:
            return ("moe_ffn_decode (AWQ-4bit, 2 <= M <= 64): alignment into blocks of 16 + gsm::awq_mma_kernel "
                    "(both GEMMs on mma.sync) + combine")
        if self.awq:
            return "moe_ffn_decode (AWQ-4bit): decode_gate_up_kernel<AWQ> + decode_down_kernel<AWQ>"
        if self.path == "grouped":
            return "moe_ffn_grouped: act_quant + gemm_kernel (both GEMMs, one persistent kernel) + combine"
        if self.routed_in_layer and self.w2_standard:
            return ("moe_ffn_decode_logits (standard W2 layout): dx1::mx_m1_kernel (top-k routing + gate/up on "
                    "mma.sync + SwiGLU + down), one kernel")
        if self.routed_in_layer:
            return "moe_ffn_decode_logits: dm::m1_kernel (top-k routing + gate/up + SwiGLU + down + combine), one kernel"
        if self.fused:
            return "moe_ffn_decode: df::fused_kernel + df::reduce_kernel, PDL-chained"
        if self.w2_standard and 2 <= self.wl.M <= 64 and self.cand:
            return ("moe_ffn_decode (standard W2 layout, 2 <= M <= 64): alignment into blocks of 16 + "
                    "gmx::mx_mma_kernel (both GEMMs on mma.sync) + combine")
        return "moe_ffn_decode: ds::gate_up_kernel + ds::down_kernel, PDL-chained"

    def launches_per_step(self) -> int:
        if self.path == "grouped":
            # (top-k), alignment, act-quant or gather, the GEMM kernel, combine
            na = 2 if self.ws_align is not None else 1
            if self.awq:
                # the b <= 16 AWQ path: one kernel for both GEMMs, then the combine
                return na + (2 if self.b <= 16 and self.cand else 3)
            return 1 + na + 3
        if self.awq:
            # fixed routing: the single-token kernel; alignment, the GEMM kernel and the
            # combine up to 64 tokens; the two decode kernels beyond
            if not self.cand:
                return 2
            return 1 if self.wl.M == 1 else (3 if self.wl.M <= 64 else 2)
        if self.w2_standard and 2 <= self.wl.M <= 64 and self.cand:
            return 4                       # top-k, alignment, the GEMM kernel, combine
        return 1 if self.routed_in_layer else 3

    def capture(self):
        with torch.cuda.stream(self.stream):
            self.launch(self.stream)            # warm, outside capture
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.launch(self.stream)
        self.stream.synchronize()
        # the layer call alone, for the roofline of the dominant kernels
        self.layer_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.layer_graph, stream=self.stream):
            self.launch_layer(self.stream)
        self.stream.synchronize()


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
    src = ("awq" if st.path == "grouped" else "awq_decode") if st.awq else st.path
    # the opt-in kernels replace some paths' kernels: their counters are keyed apart
    key = (f"{st.path}{'-w2std' if getattr(st, 'w2_standard', False) else ''}"
           f"{'-cand' if getattr(st, 'cand', False) else ''}:{wl.name}")
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


def run_ours(args, rank, world, device):
    wl = workload_from_name(args.workload)
    K, W = args.steps, args.warmup
    path, block = args.path, args.block
    if path == "auto":
        # the library's choice at the measured crossover of the two paths
        import top_moe_expert_gb300 as moe
        fmt = moe.MOE_W_AWQ4 if wl.fmt == "awq4" else moe.MOE_W_MXFP8
        p, b = moe.moe_ffn_select_path(wl.M, wl.k, wl.E, wl.d, wl.I, fmt)
        path = "decode" if p == moe.MOE_PATH_DECODE else "grouped"
        block = block or b
    st = DecodeStep(wl, K + W, device, path, block, args.w2)
    st.capture()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    s = st.stream
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(device.index if device.index is not None else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(W):
            st.x.copy_(st.x_all[i % st.n_inputs], non_blocking=True)
            st.logits.copy_(st.logits_all[i % st.n_inputs], non_blocking=True)
            flush.fill_(float(i))
            st.graph.replay()
    torch.cuda.synchronize()
    sampler.start()
    with torch.cuda.stream(s):                  # keep the GPU busy while the sampler starts
        for i in range(400):
            flush.fill_(float(i))
            st.graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(s):
        for i in range(K):
            j = (W + i) % st.n_inputs
            st.x.copy_(st.x_all[j], non_blocking=True)
            st.logits.copy_(st.logits_all[j], non_blocking=True)
            flush.fill_(float(j))
            ev0[i].record(s)
            st.graph.replay()
            ev1[i].record(s)
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    t_wall = t_wall1 - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop(t_wall0, t_wall1)
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_ms = sum(step_ms)

    # bytes of every timed step (distinct experts of that step's routing)
    bytes_steps = [step_bytes(wl, st.step_ids((W + i) % st.n_inputs)) for i in range(K)]
    total_bytes = float(sum(bytes_steps))

    # e2e: the same steps through the public API with host buffers (pinned)
    Ke = min(K, 2000)
    sel = [(W + i) % st.n_inputs for i in range(Ke)]
    # each step's inputs packed in one pinned row, laid out as st.io
    sel_rows = sel if wl.M <= 64 else list(range(st.n_inputs))
    io_pin = torch.cat([getattr(st, n)[sel_rows].reshape(len(sel_rows), -1).view(torch.uint8) for n in st.io_host],
                       dim=1).pin_memory()
    assert io_pin.shape[1] == st.io.numel()
    y_pin = torch.empty((Ke, wl.M, wl.d), dtype=torch.bfloat16).pin_memory()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(Ke):
            flush.fill_(float(i))
            e0[i].record(s)
            pi = i if wl.M <= 64 else sel[i]
            st.io.copy_(io_pin[pi], non_blocking=True)
            st.launch(s)
            y_pin[i].copy_(st.y, non_blocking=True)
            e1[i].record(s)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in zip(e0, e1))
    e2e_bytes = float(sum(bytes_steps[:Ke]))

    # the layer call alone (roofline of the dominant kernels): routing of the
    # step runs first, outside the events; L2 flushed before each call
    Kl = min(K, 2000)
    l0 = [torch.cuda.Event(enable_timing=True) for _ in range(Kl)]
    l1 = [torch.cuda.Event(enable_timing=True) for _ in range(Kl)]
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(Kl):
            j = (W + i) % st.n_inputs
            st.x.copy_(st.x_all[j], non_blocking=True)
            st.logits.copy_(st.logits_all[j], non_blocking=True)
            st.launch_pre(s)
            flush.fill_(float(j))
            l0[i].record(s)
            st.layer_graph.replay()
            l1[i].record(s)
    torch.cuda.synchronize()
    layer_ms = sum(a.elapsed_time(b) for a, b in zip(l0, l1))
    # (a layer call that routes the token itself also reads the logits)
    lb = step_bytes if st.routed_in_layer else layer_bytes
    layer_total_bytes = float(sum(lb(wl, st.step_ids((W + i) % st.n_inputs)) for i in range(Kl)))

    (total_ms, e2e_ms, layer_ms), (total_bytes, e2e_bytes, layer_total_bytes) = gather_replicas(
        [total_ms, e2e_ms, layer_ms], [total_bytes, e2e_bytes, layer_total_bytes], world, device)
    if rank != 0:
        return None

    tbps = total_bytes / (total_ms * 1e-3) / 1e12
    us_layer = total_ms * 1e3 / K
    peak_gbs, peak_kind = measured_peak()
    achieved_gbs = tbps * 1e3 / world
    line = {
        "metric": METRIC,
        "value": round(tbps, 4),
        "unit": "TB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(total_ms / K, 6),
        "us_per_layer": round(us_layer, 3),
        "tokens_per_s": round(wl.M * world / (total_ms * 1e-3 / K), 1),
        "frac_of_8TBps": round(tbps / world / 8.0, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "awq4-weights/fp16-act/f32-accum" if st.awq else "mxfp8-weights/bf16-act/f32-accum",
        "data": ("synthetic (seeded uniform 4-bit q and zeros, fp16 group scales U(0.005, 0.02), N(0,1) fp16 "
                 "activations, the fixture-A routing of the packed-AWQ study)" if st.awq else
                 "synthetic (seeded N(0,0.02) weights quantized to MXFP8, N(0,1) bf16 activations, "
                 "N(0,1) router logits; fresh routing every step)"),
        "config": {"workload": wl.name, "M": wl.M, "d": wl.d, "I": wl.I, "E": wl.E, "k": wl.k,
                   "path": ("expert-centric grouped AWQ, blocks of at most 16 rows (align + one kernel for both "
                            "GEMMs on mma.sync over the raw 4-bit codes, zero folded out in FP32 + combine, b=%d)"
                            % st.b if st.awq and st.path == "grouped" and st.b <= 16 and st.cand else
                            "expert-centric grouped AWQ (align + gather + tcgen05 kind::f16 GEMM1/GEMM2 on weights "
                            "dequantized into tensor memory + combine, b=%d)" % st.b
                            if st.awq and st.path == "grouped" else
                            ("single-token AWQ decode: gate/up + SwiGLU + down in one kernel, f16 mma.sync dot "
                             "products on raw 4-bit codes, zero folded in FP32, fixed routing") if st.awq and wl.M == 1 and st.cand else
                            ("small-batch AWQ decode (alignment into blocks of 16 + one kernel for both GEMMs on "
                             "mma.sync over the raw 4-bit codes + combine, fixed routing)")
                            if st.awq and 2 <= wl.M <= 64 and st.cand else
                            "output-centric AWQ decode (gate/up + down on CUDA cores, fixed routing)" if st.awq else
                            "expert-centric grouped (topk + align + act-quant + tcgen05 GEMM1/GEMM2 + combine, b=%d)"
                            % st.b if st.path == "grouped" else
                            ("single-token decode on the standard W2 layout: routing + gate/up + SwiGLU + down "
                             "in one kernel (mma.sync dot products)") if st.routed_in_layer and st.w2_standard else
                            "single-token decode: routing + gate/up + SwiGLU + down + combine in one kernel"
                            if st.routed_in_layer else
                            "single-pass decode (topk + fused gate/up/down + partial reduction)" if st.fused
                            else ("small-batch decode on the standard W2 layout (topk + alignment into blocks of 16 "
                                  "+ one kernel for both GEMMs on mma.sync + combine)")
                            if st.w2_standard and 2 <= wl.M <= 64 and st.cand
                            else "output-centric decode (topk + gate/up + down)") + ", CUDA graph",
                   "l2": "flushed between timed steps (512 MiB write, outside the timed interval)",
                   "parallelism": f"replicas x{world}"},
        "e2e": {"value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TB/s",
                "us_per_layer": round(e2e_ms * 1e3 / Ke, 3), "steps": Ke,
                "h2d_bytes_per_step": st.io.numel(),
                "d2h_bytes_per_step": wl.M * wl.d * 2},
        "gpu_launches": st.launches_per_step() * K,
        "roofline": roofline_obj(st, wl, layer_ms, Kl, layer_total_bytes, world),
        "clocks": clocks,
        "wall_s_timed_loop": round(t_wall, 3),
        "_path": st.path,
    }
    return line


def cpu_baseline(wl, device, path="decode", seconds=12.0):
    """The oracle, as it stands, on the host cores: steps (top-k + layer) of
    the same workload with fresh routing, on at most 4 tokens per step,
    until ~`seconds` of timed CPU work.  The oracle runs in the mode the path
    computes (exact for decode, block-scaled for grouped).  Expert weights
    are quantized by the oracle from the same fp32 draws (setup, not timed)."""
    import oracle
    from top_moe_expert_gb300 import inputs
    cache = {}

    def expert(which, e):
        if (which, e) not in cache:
            f = inputs.weights_fp32_device(wl, which, e, device).cpu().numpy().astype(np.float64)
            cache[(which, e)] = oracle.mxfp8_quantize(f)
        return cache[(which, e)]

    if wl.fmt == "awq4":
        return _cpu_baseline_awq(wl, seconds)
    mode = oracle.MODE_MX if path == "grouped" else oracle.MODE_EXACT
    S = min(wl.M, 4)
    t_total, nbytes, steps = 0.0, 0, 0
    while t_total < seconds and steps < 64:
        logits = inputs.router_logits(wl, 10_000 + steps)[:S]
        ids, _ = oracle.topk_softmax(logits, wl.k)
        experts = sorted(set(ids.reshape(-1).tolist()))
        slot = np.full(wl.E, -1, dtype=np.int32)
        slot[experts] = np.arange(len(experts), dtype=np.int32)
        ws = {}
        for which in ("w13", "w2"):
            qs = [expert(which, e) for e in experts]
            ws[which] = {"fmt": "mxfp8", "q": np.stack([q for q, _ in qs]),
                         "s": np.stack([s for _, s in qs]), "slot": slot}
        x = inputs.activations(wl, 10_000 + steps)[:S].to(torch.float64).numpy()
        t0 = time.perf_counter()
        ids2, w2 = oracle.topk_softmax(logits, wl.k)
        oracle.moe_layer(x, ids2, w2, wl.E, ws["w13"], ws["w2"], mode=mode)
        t_total += time.perf_counter() - t0
        nbytes += len(experts) * expert_bytes(wl) + S * (4 * wl.d + 4 * wl.E)
        steps += 1
    threads = min(oracle.num_threads(), S)     # the oracle parallelises over tokens
    return {"value": nbytes / t_total / 1e12, "unit": "TB/s", "cores": threads, "kind": "oracle",
            "sample": f"{steps} steps (top-k + layer, binary64, {'block-scaled' if mode else 'exact'} mode) "
                      f"of {wl.name} on {S} token(s) each, fresh routing, {t_total:.1f} s timed",
            "us_per_token": round(t_total / steps / S * 1e6, 1)}


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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_m1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "decode", "grouped"])
    ap.add_argument("--block", type=int, default=0, help="MoE block size b of the grouped path (0: automatic)")
    ap.add_argument("--w2", default="auto", choices=["auto", "standard"],
                    help="decode path: keep W2 K-contiguous (standard) instead of the neuron-major packing "
                         "small batches use by default")
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
