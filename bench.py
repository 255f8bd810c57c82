#!/usr/bin/env python
"""Benchmark of the Q4_K matmul hot path on GB300.

Default workload (`--workload decode`): one decode step = the gate/up projection
GEMV (K 5120 -> N 17408) followed by the down projection GEMV (K 17408 -> N
5120), bf16 activations, fp32 outputs, Q4_K weights drawn from N(0, 0.02^2).
The metric is effective Q4_K weight bandwidth: weight bytes streamed per second.

Other workloads (for measurement, not the headline line): `verify` (M-token
speculative-verify GEMM, K 5120 -> N 17408, --m, default 4), `prefill` (M x K
5120 -> N 17408 then M x K 17408 -> N 5120, --m, default 4096, TFLOP/s) and
`moe` (128 experts, top-8: gate, up and down with the weighted combine, --m
tokens, default 2048) and `moe_ffn` (the same layer as one routed SwiGLU expert
feed-forward call: gate, up with the SwiGLU epilogue, down on the bf16 h rows,
weighted combine), `decode_x8` (the decode step with int8 activations:
per-32 quantization of each matrix's input, then the int8 GEMV) and
`prefill_nvfp4` / `decode_nvfp4` (the prefill GEMMs and the decode GEMVs
with NVFP4 weights).

Timing: W warm-up steps, then exactly K steps between a barrier plus
cudaDeviceSynchronize on both sides, timed with CUDA events on the launching
stream.  The steps are replayed from CUDA graphs of R consecutive steps (as a
decode loop captures its layers); consecutive steps cycle through R weight sets
whose total exceeds the 129 MB L2, so the weights always come from HBM.  SM clocks and throttle reasons are sampled through NVML
during the timed region.  `e2e` repeats the metric through the public API with
the activations copied from pinned host memory and the outputs copied back every
step.  `--impl reference` times the plain-C oracle on the host cores instead.

Under torchrun each rank runs the same workload on its own GPU (independent
replicas, weak scaling); the reported time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4_K matmul effective weight GB/s (decode) and TFLOP/s (prefill) vs roofline"
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
L2_BYTES = 129 * 10 ** 6


# ------------------------------------------------------------------ helpers

def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), \
        int(os.environ.get("WORLD_SIZE", "1"))


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The maximum of a per-rank time over all ranks (each rank is an independent
    replica; the job is as slow as its slowest rank).  World size 1: v itself."""
    if world <= 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(per_step_value: float, world: int) -> float:
    """Whole-job throughput: every rank processes the same per-step work (weak
    scaling), so the job's value is the per-rank value at the max-over-ranks time
    times the number of ranks."""
    return per_step_value * world


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, FALLBACK_BF16_TFLOPS, "fallback"


def source_sha(rel: str) -> str:
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel's source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)[kernel]
        if d["source_sha256"] != source_sha(d["source"]):
            return None
        return float(d["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """Samples SM clock, max clock and clock-event reasons via NVML (read only)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, cuda_index: int):
        self.samples, self.reasons, self.max_mhz, self.power_mw = [], 0, None, []
        self._stop = threading.Event()
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            ok = False
            try:
                import torch
                props = torch.cuda.get_device_properties(cuda_index)
                bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[cuda_index]) if vis and vis.split(",")[0].isdigit() else cuda_index
                if nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                    return
            self._nvml, self._h = nv, h
            m = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = m.value
        except OSError:
            self._nvml = None

    def _run(self):
        nv, h = self._nvml, self._h
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if get_reasons(h, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            if nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(c)) == 0:
                self.power_mw.append(c.value)
            time.sleep(0.005)

    def __enter__(self):
        if self._nvml is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self._nvml is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"]}
        out = {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
               "reasons": [n for b, n in self.REASONS.items() if self.reasons & b and n != "gpu_idle"],
               "samples": len(self.samples)}
        if self.power_mw:
            out["power_w"] = statistics.median(self.power_mw) / 1e3
        return out


# --------------------------------------------------------------- workloads

# the expert weights do not depend on the token count: generated once per process
_MOE_WEIGHTS = {}


class Workload:
    """Holds the host inputs of one workload and knows how to run one step."""

    def __init__(self, name: str, m: int):
        import numpy as np
        import synth
        self.name, self.m = name, m
        self.np = np
        self.mats = []   # list of (tag, N, K, M, blocks, x) for dense GEMM steps
        self.moe = None
        self.x8 = name == "decode_x8"
        self.fp4 = {}  # NVFP4 workloads: tag -> tensor scale g
        if name in ("decode", "decode_x8"):
            mt = m if self.x8 else 1  # the int8 variant also runs at verify sizes (--m up to 16)
            self.mats = [("gate_up", 17408, 5120, mt, synth.weights(synth.seed(1, 0), 17408, 5120),
                          synth.normal_bf16(synth.seed(1, 1), mt * 5120).reshape(mt, 5120)),
                         ("down", 5120, 17408, mt, synth.weights(synth.seed(1, 5), 5120, 17408),
                          synth.normal_bf16(synth.seed(1, 6), mt * 17408).reshape(mt, 17408))]
            self.unit, self.config = "GB/s", {"workload": "decode GEMV M=1: K5120->N17408 then K17408->N5120"}
            if self.x8:
                self.config = {"workload": f"decode GEMV M={mt} with int8 activations (per-32 scales, quantized "
                                           "in the step): K5120->N17408 then K17408->N5120"}
                self.mats = [(tag + "_x8",) + tuple(rest) for (tag, *rest) in self.mats]
        elif name == "verify":
            self.mats = [("verify", 17408, 5120, m, synth.weights(synth.seed(2, 0), 17408, 5120),
                          synth.normal_bf16(synth.seed(2, 1), m * 5120).reshape(m, 5120))]
            self.unit, self.config = "GB/s", {"workload": f"speculative-verify GEMM M={m}: K5120->N17408"}
        elif name == "prefill":
            self.mats = [("prefill_up", 17408, 5120, m, synth.weights(synth.seed(3, 0), 17408, 5120, 0.02, 0.01,
                                                                       10.0, synth.seed(3, 4)),
                          synth.normal_bf16(synth.seed(3, 1), m * 5120).reshape(m, 5120)),
                         ("prefill_down", 5120, 17408, m, synth.weights(synth.seed(3, 5), 5120, 17408, 0.02, 0.01,
                                                                         10.0, synth.seed(3, 9)),
                          synth.normal_bf16(synth.seed(3, 6), m * 17408).reshape(m, 17408))]
            self.unit, self.config = "TFLOP/s", {"workload": f"prefill GEMM M={m}: K5120->N17408 then K17408->N5120"}
        elif name == "decode_nvfp4":
            mats = []
            for tag, N, K, sw, sx in (("gate_up_fp4", 17408, 5120, 10, 11), ("down_fp4", 5120, 17408, 12, 13)):
                blocks, g = synth.nvfp4_weights(synth.seed(8, sw), N, K)
                self.fp4[tag] = float(g)
                mats.append((tag, N, K, m, blocks, synth.normal_bf16(synth.seed(8, sx), m * K).reshape(m, K)))
            self.mats = mats
            self.unit, self.config = "GB/s", {"workload": f"decode GEMV M={m} with NVFP4 weights: K5120->N17408 "
                                                          "then K17408->N5120"}
        elif name == "prefill_nvfp4":
            mats = []
            for tag, N, K, sw, sx in (("prefill_up_fp4", 17408, 5120, 0, 1), ("prefill_down_fp4", 5120, 17408, 5, 6)):
                blocks, g = synth.nvfp4_weights(synth.seed(8, sw), N, K)
                self.fp4[tag] = float(g)
                mats.append((tag, N, K, m, blocks, synth.normal_bf16(synth.seed(8, sx), m * K).reshape(m, K)))
            self.mats = mats
            self.unit, self.config = "TFLOP/s", {"workload": f"prefill GEMM with NVFP4 weights M={m}: "
                                                             "K5120->N17408 then K17408->N5120"}
        elif name in ("moe", "moe_ffn"):
            E, topk = 128, 8
            ids, gates = synth.routing(synth.seed(4, 2) + m, synth.seed(4, 3) + m, m, E, topk)
            mk = lambda s, N, K: _MOE_WEIGHTS.setdefault((s, N, K), np.concatenate(  # noqa: E731
                [synth.weights(synth.seed(4, s) + 1000 * (e + 1), N, K) for e in range(E)]))
            self.moe = dict(E=E, topk=topk, T=m, ids=ids, gates=gates, ffn=name == "moe_ffn",
                            gate=mk(0, 768, 2048), up=mk(7, 768, 2048), down=mk(5, 2048, 768),
                            x=synth.normal_bf16(synth.seed(4, 1), m * 2048).reshape(m, 2048),
                            xd=synth.normal_bf16(synth.seed(4, 6), m * topk * 768).reshape(m * topk, 768))
            self.unit, self.config = "GB/s", {"workload": f"MoE 128 experts top-8 T={m}: gate+up K2048->N768 "
                                                          "per slot, down K768->N2048 with weighted combine"}
            if name == "moe_ffn":
                self.config = {"workload": f"routed SwiGLU expert FFN, 128 experts top-8 T={m}: gate+up "
                                           "K2048->H768, SwiGLU to bf16, down K768->D2048, weighted combine"}
        else:
            raise SystemExit(f"unknown workload {name}")

    # algorithmic quantities per step
    def weight_bytes(self) -> float:
        if self.moe:
            touched = len(set(self.moe["ids"].reshape(-1).tolist()))
            return touched * (2 * 768 * 2048 + 2048 * 768) * 144 / 256
        return float(sum(N * K * 144 // 256 for _, N, K, *_ in self.mats))

    def flops(self) -> float:
        if self.moe:
            items = self.moe["T"] * self.moe["topk"]
            return 2.0 * items * 3 * 768 * 2048
        return float(sum(2 * M * N * K for _, N, K, M, *_ in self.mats))

    def value(self, seconds_per_step: float) -> float:
        if self.unit == "TFLOP/s":
            return self.flops() / seconds_per_step / 1e12
        return self.weight_bytes() / seconds_per_step / 1e9


class DeviceRunner:
    """Device buffers (R rotating weight sets) and per-step launch functions."""

    def __init__(self, wl: Workload, device):
        import torch
        import q4_weight_quantized_gb300 as q4k
        self.torch, self.q4k, self.wl, self.dev = torch, q4k, wl, device
        self.sh = None  # the stream handle every call is enqueued on (None: torch's current stream)
        np = wl.np

        def d(a):
            a = np.ascontiguousarray(a)
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(device)

        per_set = wl.weight_bytes() if not wl.moe else sum(wl.moe[k].nbytes for k in ("gate", "up", "down"))
        self.R = max(2, int(4 * L2_BYTES // per_set) + 1)
        if wl.moe:
            self.R = max(2, min(self.R, 6))
        self.sets, self.x, self.y, self.ws = [], [], [], []
        if wl.moe:
            mo = wl.moe
            base = {k: d(mo[k]) for k in ("gate", "up", "down")}
            for r in range(self.R):
                self.sets.append(base if r == 0 else {k: v.clone() for k, v in base.items()})
            self.ids, self.gates = d(mo["ids"]), d(mo["gates"])
            self.xg, self.xd = d(mo["x"]), d(mo["xd"])
            T, topk = mo["T"], mo["topk"]
            self.y_gate = torch.empty((T, topk, 768), dtype=torch.float32, device=device)
            self.y_up = torch.empty((T, topk, 768), dtype=torch.float32, device=device)
            self.y_down = torch.empty((T, 2048), dtype=torch.float32, device=device)
            wsb = max(q4k.q4k_moe_workspace_size(mo["E"], 768, 2048, T, topk, 0),
                      q4k.q4k_moe_workspace_size(mo["E"], 2048, 768, T, topk, 1),
                      q4k.q4k_moe_ffn_workspace_size(mo["E"], 768, 2048, T, topk))
            self.moe_ws = torch.empty(wsb, dtype=torch.uint8, device=device)
            self.moe_wsb = wsb
        else:
            base = [d(b) for (_, _, _, _, b, _) in wl.mats]
            for r in range(self.R):
                self.sets.append(base if r == 0 else [t.clone() for t in base])
            self.q, self.sx = [], []
            # a step's activations and outputs each live in one buffer (matrix i's rows
            # are a view into it), so that end to end a step is one copy in and one out
            nx = [M * K for (_, N, K, M, _, _) in wl.mats]
            ny = [M * N for (_, N, K, M, _, _) in wl.mats]
            self.x_all = torch.empty(sum(nx), dtype=torch.int16, device=device)
            self.y_all = torch.empty(sum(ny), dtype=torch.float32, device=device)
            ox = oy = 0
            for i, (_, N, K, M, _, x) in enumerate(wl.mats):
                xv = self.x_all[ox:ox + nx[i]].view(M, K)
                xv.copy_(d(x))
                self.x.append(xv)
                self.y.append(self.y_all[oy:oy + ny[i]].view(M, N))
                ox += nx[i]
                oy += ny[i]
                if wl.x8:
                    self.q.append(torch.empty((M, K), dtype=torch.int8, device=device))
                    self.sx.append(torch.empty((M, K // 32), dtype=torch.float32, device=device))
                wsb = q4k.q4k_gemm_workspace_size(M, N, K)
                self.ws.append((torch.empty(max(wsb, 1), dtype=torch.uint8, device=device), wsb))

    def launches_per_step(self) -> int:
        if self.wl.moe:
            mo = self.wl.moe
            # one routing (none for up to 16 items); per grouped GEMM the expert GEMM
            # (+ the activation gather on the tensor-core path, from 32 items per
            # expert; the FFN call gathers once); + the combine
            items = mo["T"] * mo["topk"]
            tc = items >= 32 * mo["E"]
            route = 1 if (tc or items > 16) else 0
            if mo["ffn"]:
                return route + (1 if tc else 0) + 3 + 1
            return route + 3 * (2 if tc else 1) + 1
        return len(self.wl.mats) * (2 if self.wl.x8 else 1)  # per matrix: (quantize +) GEMV

    def step_one(self, r: int, i: int):
        """Enqueue only matrix i of the step, with weight set r."""
        q4k, wl = self.q4k, self.wl
        tag, N, K, M, _, _ = wl.mats[i]
        if tag in wl.fp4:
            q4k.q4k_nvfp4_gemm(self.sets[r][i], wl.fp4[tag], N, K, self.x[i], M, K, self.y[i], N, stream=self.sh)
        elif wl.x8:
            q4k.q4k_gemm_x8(self.sets[r][i], N, K, self.q[i], self.sx[i], M, self.y[i], N, None, 0, stream=self.sh)
        elif M == 1:
            q4k.q4k_gemv(self.sets[r][i], N, K, self.x[i], self.y[i], stream=self.sh)
        else:
            ws, wsb = self.ws[i]
            q4k.q4k_gemm(self.sets[r][i], N, K, self.x[i], M, K, self.y[i], N, ws if wsb else None, wsb, stream=self.sh)

    def kernel_calls(self):
        """(tag, enqueue(r)) for each separately timed kernel of the step.  Dense:
        each matrix's GEMM.  MoE: the up projection call on the routing the step left
        in the workspace (the expert GEMM; on the tensor-core path, from 32 items per
        expert, the activation gather it starts with is inside the call too)."""
        if self.wl.moe:
            mo, q4k = self.wl.moe, self.q4k
            E, T, topk = mo["E"], mo["T"], mo["topk"]

            def up(r):
                q4k.q4k_moe_grouped_gemm_reuse_routing(self.sets[r]["up"], E, 768, 2048, self.xg, 0, self.ids,
                                                       self.gates, T, topk, self.y_up, 0, self.moe_ws, self.moe_wsb,
                                                       stream=self.sh)
            return [("moe_up", up)]
        return [(tag, (lambda r, i=i: self.step_one(r, i))) for i, (tag, *_) in enumerate(self.wl.mats)]

    def kernel_roofline(self, tag: str):
        """Algorithmic work of one launch of kernel `tag`: ("hbm", bytes) or ("tensor", flops)."""
        wl = self.wl
        if wl.moe:
            mo = wl.moe
            items = mo["T"] * mo["topk"]
            if items >= 32 * mo["E"]:
                return "tensor", 2.0 * items * 768 * 2048
            touched = len(set(mo["ids"].reshape(-1).tolist()))
            return "hbm", touched * 768 * 2048 * 144 / 256 + mo["T"] * 2048 * 2 + items * 768 * 4
        _, N, K, M, *_ = next(m for m in wl.mats if m[0] == tag)
        if wl.unit == "TFLOP/s":
            return "tensor", 2.0 * M * N * K
        return "hbm", N * K * 144 / 256 + (M * K + M * K // 32 * 4 if wl.x8 else M * K * 2) + M * N * 4

    def step(self, r: int, mark=None):
        """Enqueue one step using weight set r.  mark(i) is called before
        matrix i and after the last one (to record events)."""
        q4k, wl = self.q4k, self.wl
        if wl.moe:
            mo, s = wl.moe, self.sets[r]
            E, T, topk = mo["E"], mo["T"], mo["topk"]
            if mark:
                mark(0)
            if mo["ffn"]:
                q4k.q4k_moe_ffn(s["gate"], s["up"], s["down"], E, 768, 2048, self.xg, self.ids, self.gates, T, topk,
                                self.y_down, self.moe_ws, self.moe_wsb, stream=self.sh)
                if mark:
                    mark(1)
                return
            # the layer's three projections share one routing: the first call sorts
            # the items, the other two reuse the sort left in the workspace
            q4k.q4k_moe_grouped_gemm(s["gate"], E, 768, 2048, self.xg, 0, self.ids, self.gates, T, topk, self.y_gate,
                                     0, self.moe_ws, self.moe_wsb, stream=self.sh)
            q4k.q4k_moe_grouped_gemm_reuse_routing(s["up"], E, 768, 2048, self.xg, 0, self.ids, self.gates, T, topk,
                                                   self.y_up, 0, self.moe_ws, self.moe_wsb, stream=self.sh)
            q4k.q4k_moe_grouped_gemm_reuse_routing(s["down"], E, 2048, 768, self.xd, 1, self.ids, self.gates, T, topk,
                                                   self.y_down, 1, self.moe_ws, self.moe_wsb, stream=self.sh)
            if mark:
                mark(1)
            return
        for i, (tag, N, K, M, _, _) in enumerate(wl.mats):
            if mark:
                mark(i)
            if tag in wl.fp4:
                q4k.q4k_nvfp4_gemm(self.sets[r][i], wl.fp4[tag], N, K, self.x[i], M, K, self.y[i], N, stream=self.sh)
            elif wl.x8:
                q4k.q4k_quantize_x8(self.x[i], M, K, K, self.q[i], self.sx[i], stream=self.sh)
                q4k.q4k_gemm_x8(self.sets[r][i], N, K, self.q[i], self.sx[i], M, self.y[i], N, None, 0,
                                stream=self.sh)
            elif M == 1:
                q4k.q4k_gemv(self.sets[r][i], N, K, self.x[i], self.y[i], stream=self.sh)
            else:
                ws, wsb = self.ws[i]
                q4k.q4k_gemm(self.sets[r][i], N, K, self.x[i], M, K, self.y[i], N, ws if wsb else None, wsb, stream=self.sh)
        if mark:
            mark(len(wl.mats))


def measure(wl, args, steps, warmup, stream, device, world, e2e=True):
    """Times `steps` steps of workload `wl` on `stream` (after `warmup` untimed
    steps); returns the record for the JSON line: value, time per step, the
    dominant kernel's roofline, per-kernel times, clocks, spread and (e2e) the
    end-to-end figure through the public API."""
    import numpy as np
    import torch
    import torch.distributed as dist
    import q4_weight_quantized_gb300 as q4k

    gr = DeviceRunner(wl, device)
    gr.sh = stream.cuda_stream  # every call names its stream, as a serving loop would

    # warm the host-side state (descriptors, attributes) before capture
    with torch.cuda.stream(stream):
        for r in range(gr.R):
            gr.step(r)
    torch.cuda.synchronize()
    q4k.q4k_check_device(stream)

    # Steps are captured R at a time (step r uses weight set r), as a decode loop
    # captures its layers: one graph of R consecutive steps, replayed, plus one
    # graph of the first K mod R (and W mod R) steps, so that exactly K timed
    # and W warm-up steps run.  Nothing else is in the graphs.
    def capture(n):
        if n == 0:
            return None
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(n):
                gr.step(r)
        return g

    g_full = capture(gr.R)
    g_rem = capture(steps % gr.R)
    g_wrem = capture(warmup % gr.R)

    def run_steps(n, rem):
        for _ in range(n // gr.R):
            g_full.replay()
        if rem is not None:
            rem.replay()

    # warm-up steps
    with torch.cuda.stream(stream):
        run_steps(warmup, g_wrem)
    torch.cuda.synchronize()

    # timed region
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(device.index)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clocks:
        with torch.cuda.stream(stream):
            t0.record(stream)
            run_steps(steps, g_rem)
            t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = t0.elapsed_time(t1)
    q4k.q4k_check_device(stream)

    # spread: a separate pass of graph replays, each bracketed by events, so that the
    # events do not touch the timed region above
    n_rep = max(3, min(200, steps // gr.R))
    with torch.cuda.stream(stream):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_rep + 1)]
        evs[0].record(stream)
        for i in range(n_rep):
            g_full.replay()
            evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = sorted(evs[i].elapsed_time(evs[i + 1]) / gr.R for i in range(n_rep))
    spread = {"replays": n_rep, "steps_per_replay": gr.R, "median_ms_per_step": statistics.median(per),
              "best_ms_per_step": per[0], "worst_ms_per_step": per[-1]}

    # per-kernel durations: each kernel of the step alone, R launches over the R
    # weight sets per graph, replayed back to back and timed with CUDA events on
    # the launching stream (average launch duration, launch gaps included)
    kernel_ms = {}
    for tag, call in gr.kernel_calls():
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(gr.R):
                call(r)
        reps = max(3, min(200, steps // gr.R))
        with torch.cuda.stream(stream):
            g.replay()
            k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            k0.record(stream)
            for _ in range(reps):
                g.replay()
            k1.record(stream)
        torch.cuda.synchronize()
        kernel_ms[tag] = k0.elapsed_time(k1) / (reps * gr.R)
    q4k.q4k_check_device(stream)

    ms = max_over_ranks(ms, world, device)

    # end to end through the public API: activations from pinned host memory,
    # outputs back to pinned host memory, every step
    e2e_rec = None
    if e2e and not wl.moe:
        hx = torch.from_numpy(np.concatenate([np.ascontiguousarray(x).view(np.int16).reshape(-1)
                                              for (*_, x) in wl.mats])).pin_memory()
        hy = torch.empty(gr.y_all.shape, dtype=torch.float32).pin_memory()
        e2e_steps = min(steps, 2000)
        with torch.cuda.stream(stream):
            for i in range(10):
                gr.x_all.copy_(hx, non_blocking=True)
                gr.step(i % gr.R)
                hy.copy_(gr.y_all, non_blocking=True)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(e2e_steps):
                gr.x_all.copy_(hx, non_blocking=True)  # the step's activations, pinned host -> device
                gr.step(i % gr.R)
                hy.copy_(gr.y_all, non_blocking=True)  # the step's outputs, device -> pinned host
            e1.record(stream)
            torch.cuda.synchronize()
        ems = e0.elapsed_time(e1)
        ems = max_over_ranks(ems, world, device)
        # the same steps captured into CUDA graphs (R steps per graph), each step its
        # pinned host -> device copy, the public API calls and the device -> host copy,
        # as a serving loop replays its captured layers: the library without the host
        # issue cost of a Python loop
        gg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gg, stream=stream):
            for r in range(gr.R):
                gr.x_all.copy_(hx, non_blocking=True)
                gr.step(r)
                hy.copy_(gr.y_all, non_blocking=True)
        g_steps = max(gr.R, (e2e_steps // gr.R) * gr.R)
        with torch.cuda.stream(stream):
            for _ in range(3):
                gg.replay()
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            e0.record(stream)
            for _ in range(g_steps // gr.R):
                gg.replay()
            e1.record(stream)
            torch.cuda.synchronize()
        gms = max_over_ranks(e0.elapsed_time(e1), world, device)
        e2e_rec = {"value": job_value(wl.value(gms / 1e3 / g_steps), world), "unit": wl.unit,
                   "h2d_bytes_per_step": int(hx.numel() * 2), "d2h_bytes_per_step": int(hy.numel() * 4),
                   "steps": g_steps,
                   "how": "CUDA graphs of %d steps, each: pinned host->device copy of the step's activations, the "
                          "public API calls, device->host copy of its outputs" % gr.R,
                   "eager": {"value": job_value(wl.value(ems / 1e3 / e2e_steps), world), "steps": e2e_steps,
                             "how": "the same per step from a Python loop (host issue bound)"}}

    hbm, bf16, bf16_s, src = peaks()
    sec_per_step = ms / 1e3 / steps
    rec = {
        "value": job_value(wl.value(sec_per_step), world), "unit": wl.unit, "steps": steps, "warmup": warmup,
        "ms_per_step": ms / steps,
        "config": dict(wl.config, l2="rotating %d weight sets, %.0f MB total > 129 MB L2" %
                       (gr.R, gr.R * (wl.weight_bytes() if not wl.moe else sum(
                           wl.moe[k].nbytes for k in ("gate", "up", "down"))) / 1e6),
                       parallelism="replicas x%d" % world, static_weights=True,
                       timing="CUDA graphs of %d steps, CUDA events; kernel times from per-kernel graphs" % gr.R),
        "gpu_launches": gr.launches_per_step() * steps,
    }
    # roofline of the dominant (slowest) kernel
    tag = max(kernel_ms, key=kernel_ms.get)
    bound, algo = gr.kernel_roofline(tag)
    sec = kernel_ms[tag] / 1e3
    if bound == "tensor":
        ach = algo / sec / 1e12
        rec["roofline"] = {"bound": "tensor", "achieved": ach, "peak": bf16, "unit": "TFLOP/s", "frac": ach / bf16,
                           "traffic": profiled_traffic(tag), "kernel": tag, "kernel_us": kernel_ms[tag] * 1e3,
                           "algorithmic_flops": algo, "peak_source": src + " (burst)"}
    else:
        ach = algo / sec / 1e9
        rec["roofline"] = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                           "traffic": profiled_traffic(tag), "kernel": tag, "kernel_us": kernel_ms[tag] * 1e3,
                           "algorithmic_bytes": algo, "peak_source": src, "frac_of_nominal_8tbs": ach / 8000.0}
    rec["kernels_us"] = {k: v * 1e3 for k, v in kernel_ms.items()}
    rec["clocks"] = clocks.summary()
    rec["spread"] = spread
    if e2e_rec:
        rec["e2e"] = e2e_rec
    del gr
    torch.cuda.empty_cache()
    return rec


# the other configurations, measured in the default run beside the decode
# headline: (key, workload, tokens)
SUB_WORKLOADS = (("verify_m4", "verify", 4), ("prefill_m4096", "prefill", 4096), ("prefill_m128", "prefill", 128),
                 ("moe_t16", "moe", 16), ("moe_t2048", "moe", 2048))


def run_gpu(args, rank, local_rank, world):
    import torch
    import torch.distributed as dist
    from q4_weight_quantized_gb300.build import build_library
    import q4_weight_quantized_gb300 as q4k

    build_library()
    q4k.load()
    # weights are uploaded once and only read afterwards, as in serving: the
    # small-M kernels may copy their first weight blocks while the previous
    # kernel drains (include/q4k.h, q4k_set_static_weights)
    q4k.q4k_set_static_weights(True)
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    stream = torch.cuda.Stream(device)

    wl = Workload(args.workload, args.m)
    rec = measure(wl, args, args.steps, args.warmup, stream, device, world, e2e=True)
    line = {"metric": METRIC, "value": rec["value"], "unit": rec["unit"], "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("int8 (per-32 fp32 scales) x Q4_K -> fp32" if wl.x8 else
                      "bf16 x NVFP4 -> fp32" if wl.fp4 else "bf16 x Q4_K -> fp32"),
            "data": "synthetic (seeded N(0,0.02^2) weights quantized to Q4_K; N(0,1) bf16 activations)"}
    for k in ("config", "gpu_launches", "roofline", "kernels_us", "clocks", "spread", "e2e"):
        if k in rec:
            line[k] = rec[k]
    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)

    # every other configuration, each timed the same way with its own step count
    # (about half a second of timed work, at most --steps)
    if args.workload == "decode" and not args.no_workloads:
        subs = {}
        for key, name, m in SUB_WORKLOADS:
            swl = Workload(name, m)
            est = swl.flops() / 1.0e15 if swl.unit == "TFLOP/s" else swl.weight_bytes() / 4.0e12
            if swl.moe:
                est = max(est, 2.0 * swl.flops() / 1.0e15)
            n = int(max(2 * args.warmup, min(args.steps, 0.5 / max(est, 1e-6))))
            r = measure(swl, args, n, args.warmup, stream, device, world, e2e=False)
            r["config"] = dict(r["config"])
            if rank == 0 and not args.no_cpu:
                r["cpu_baseline"] = cpu_baseline(swl, budget_s=max(2.0, args.cpu_seconds / 3))
            subs[key] = r
        line["workloads"] = subs
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------ oracle (CPU)

def cpu_baseline(wl: Workload, budget_s: float = 8.0):
    """Times the oracle (as it stands) on the host cores over the same inputs, for
    about `budget_s` seconds, in the workload's own unit.  Dense workloads run the
    whole step while that fits the budget, else a sample of each matrix's rows
    (every token); the MoE layer runs whole, or on a sample of its tokens.  A
    sampled figure is the work done divided by the time taken, which is what the
    full workload would give at the same rate."""
    import oracle
    oracle.build()
    np = wl.np
    threads = os.cpu_count() or 1
    if wl.moe:
        mo = wl.moe
        E, T, topk = mo["E"], mo["T"], mo["topk"]
        def layer(n):  # the layer's three projections over the first n tokens
            ids, gates = mo["ids"][:n], mo["gates"][:n]
            x, xd = mo["x"][:n], mo["xd"][:n * topk]
            t = time.perf_counter()
            oracle.moe(mo["gate"], E, 768, 2048, x, False, ids, threads=threads)
            oracle.moe(mo["up"], E, 768, 2048, x, False, ids, threads=threads)
            oracle.moe(mo["down"], E, 2048, 768, xd, True, ids, gates, threads=threads)
            return time.perf_counter() - t

        n0 = min(T, 4)
        per_token = layer(n0) / n0  # calibration, not counted
        t_sample = int(max(1, min(T, budget_s / 3 / max(per_token, 1e-9))))
        done_tokens, t_total, reps = 0, 0.0, 0
        while t_total < budget_s:
            t_total += layer(t_sample)
            done_tokens += t_sample
            reps += 1
        sec_per_layer = t_total / done_tokens * T
        sample = (f"{reps} layer passes over {t_sample} of the {T} tokens, {t_total:.1f} s, time per layer "
                  f"projected from the time per token; plain C, fp64 accumulate, {threads} pthreads")
        value = wl.value(sec_per_layer)
        return {"value": value, "unit": wl.unit, "cores": threads, "kind": "oracle", "sample": sample}
    # dense: rows per matrix so that one pass over all matrices takes about a third
    # of the budget (all rows when that fits)
    t = time.perf_counter()
    for (_, N, K, M, blocks, x) in wl.mats:
        oracle.gemm(np.ascontiguousarray(blocks[:16]), 16, K, x, threads=threads)
    per_row = (time.perf_counter() - t) / 16
    rows = [max(1, min(N, int(budget_s / 3 / max(per_row, 1e-9) / len(wl.mats)))) for (_, N, *_) in wl.mats]
    subs = [(np.ascontiguousarray(b[:n]) if n < N else b, n, K, M, x)
            for (n, (_, N, K, M, b, x)) in zip(rows, wl.mats)]
    done, t_total, reps = 0.0, 0.0, 0
    while t_total < budget_s:
        for (b, n, K, M, x) in subs:
            t = time.perf_counter()
            oracle.gemm(b, n, K, x, threads=threads)
            t_total += time.perf_counter() - t
            done += 2.0 * M * n * K if wl.unit == "TFLOP/s" else n * K * 144 / 256
        reps += 1
    value = done / t_total / (1e12 if wl.unit == "TFLOP/s" else 1e9)
    full = all(n == N for n, (_, N, *_) in zip(rows, wl.mats))
    what = "all rows" if full else "rows " + " and ".join(f"{n} of {N}" for n, (_, N, *_) in zip(rows, wl.mats))
    return {"value": value, "unit": wl.unit, "cores": threads, "kind": "oracle",
            "sample": f"{reps} passes over {what} of each matrix, every token, {t_total:.1f} s, plain C, "
                      f"fp64 accumulate, rows split over {threads} pthreads"}


def run_reference(args, rank, world):
    """--impl reference: the oracle on the host cores, same metric and workload;
    each step is a bounded row sample of the decode step."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = Workload(args.workload if args.workload in ("decode", "verify") else "decode", args.m)
    np = wl.np
    threads = os.cpu_count() or 1
    # calibrate a row sample so that warm-up + steps take about two minutes
    t = time.perf_counter()
    for (_, N, K, M, blocks, x) in wl.mats:
        oracle.gemm(np.ascontiguousarray(blocks[:256]), 256, K, x, threads=threads)
    per_row = (time.perf_counter() - t) / 256 / len(wl.mats)
    budget_per_step = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(1, min(min(N for _, N, *_ in wl.mats), budget_per_step / max(per_row, 1e-9) / len(wl.mats))))
    subs = [(np.ascontiguousarray(b[:rows]), K, x) for (_, N, K, M, b, x) in wl.mats]

    def step():
        nbytes = 0
        for (b, K, x) in subs:
            oracle.gemm(b, rows, K, x, threads=threads)
            nbytes += rows * K * 144 / 256
        return nbytes

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(args.steps):
        total += step()
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    sample = f"{rows} rows of each matrix per step ({args.steps} steps), plain C oracle, {threads} pthreads"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": wl.unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32 dequant, fp64 accumulate",
            "data": "synthetic (seeded, same inputs as the GPU arm)", "config": wl.config,
            "cpu_baseline": {"value": value, "unit": wl.unit, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": wl.unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["decode", "decode_x8", "decode_nvfp4", "verify", "prefill",
                                           "prefill_nvfp4", "moe", "moe_ffn"],
                    default="decode")
    ap.add_argument("--m", type=int, default=None, help="tokens (verify: 4, prefill: 4096, moe: 2048)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the cpu_baseline legs")
    ap.add_argument("--no-workloads", action="store_true",
                    help="decode: skip the other configurations' records (verify, prefill, MoE)")
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    args = ap.parse_args()
    if args.m is None:
        args.m = {"decode": 1, "decode_x8": 1, "decode_nvfp4": 1, "verify": 4, "prefill": 4096, "prefill_nvfp4": 4096, "moe": 2048,
                  "moe_ffn": 2048}[args.workload]
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, local_rank, world = env_rank()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, local_rank, world)


if __name__ == "__main__":
    main()
