#!/usr/bin/env python3
"""Benchmark of the quantized projection path on GB300.

Default run (N = 1): the 27B-class decode layer at B = 1 (hidden 5120; q, k,
v, o projections, paired gate/up 5120 -> 2x17408, down 17408 -> 5120, each
input produced by the fused RMSNorm + Q8_1 kernel) -- reported as HBM GB/s --
and the same layer's 512-token prefill (all seven projections through the
tensor-core GEMM) -- reported as effective int8-op TOPS -- in one JSON line.

A step is one pass of the whole path over one batch: every RMSNorm+Q8_1 and
every projection of the layer.  Inputs are synthetic (seeded generators of
gemm_zq_rmsnorm_gb300.inputs), resident in HBM before timing.  L2 (129 MB)
is defeated by rotating distinct copies of the weights (>= 3x L2 per
rotation).  Steps are replayed from CUDA graphs; timing is CUDA events on the
launching stream, W warm-up steps, K timed steps, max over ranks.

--impl reference times the CPU oracle (the only other implementation of this
path) on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gemm_zq_rmsnorm_gb300 import inputs  # noqa: E402

METRIC = "Q4_K GEMV HBM GB/s (B=1) & GEMM int8 TOPS (B=512), % of GB300 roofline"
L2_BYTES = 129 * 1024 * 1024


def recorded_traffic(key):
    """DRAM bytes per launch from the committed ncu capture (profiles/traffic.json),
    or None when the kernel source changed since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(key)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != rec["sha256_16"]:
        return None
    return int(rec["dram_bytes"])


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
def input_key(pname):
    """Projections that read the same normalised input share one RMSNorm+Q8_1."""
    return {"q_proj": "attn", "k_proj": "attn", "v_proj": "attn", "o_proj": "o",
            "gate_up": "ffn", "down": "down"}.get(pname, pname)


def layer_inputs(shapes):
    seen = []
    for (pname, K, N, paired) in shapes:
        if input_key(pname) not in [k for k, _ in seen]:
            seen.append((input_key(pname), K))
    return seen


def layer_algo_bytes(shapes, B, layers=1, extra=()):
    """Algorithmic bytes of one step: each RMSNorm+Q8_1 (x read, Q8_1 written)
    and each projection (weights once, its Q8_1 input once -- a pair reads it
    once for both matrices at B = 1 --, fp32 outputs)."""
    b = sum(norm_bytes(K, B) for _, K in layer_inputs(shapes))
    for (pname, K, N, paired) in list(shapes) * layers + list(extra):
        b += proj_bytes(K, N, B) * (2 if paired else 1) - (B * K * (1 + 4 / 32) if paired and B == 1 else 0)
    return b


def rotation_copies(shapes, layers=1, extra=(), min_rotation_bytes=3 * L2_BYTES):
    """Distinct weight copies a benchmark rotates through so that each step
    reads its weights from HBM, not from L2."""
    per_copy = (sum(N * K * 144 // 256 * (2 if p else 1) for (_, K, N, p) in shapes) * layers
                + sum(N * K * 144 // 256 * (2 if p else 1) for (_, K, N, p) in extra))
    return max(1, -(-min_rotation_bytes // per_copy))


def decode_config(name, shapes, layers=1, extra=(), R=None, fused=True, prefetch=False):
    """The `config` of a B = 1 decode line (both arms print the same one)."""
    R = rotation_copies(shapes, layers, extra) if R is None else R
    return {"workload": name, "B": 1, "hidden": layer_inputs(shapes)[0][1],
            "projections": [f"{p} {K}->{N}{' x2' if pr else ''}" for (p, K, N, pr) in list(shapes) + list(extra)],
            "layers": layers, "weight_copies_rotated": R,
            "decode_path": ("fused: one launch per layer input (RMSNorm + Q8_1 in the mat-vec kernel)"
                            + ("; each launch pulls the next one's weights into L2" if prefetch else "")
                            if fused else "two-step: RMSNorm+Q8_1, then one launch per projection"),
            "l2": f"inputs larger than L2: {R} rotating weight copies of the step",
            "algorithmic_bytes_per_step": int(layer_algo_bytes(shapes, 1, layers, extra))}


def proj_bytes(K, N, B):
    """Algorithmic bytes of one projection: weights once, Q8_1 input, fp32 y."""
    return N * K * 144 // 256 + B * K * (1 + 4 / 32) + B * N * 4


def norm_bytes(K, B):
    return B * K * 4 + B * K * (1 + 4 / 32)


class LayerWorkload:
    """One decoder layer's projections at batch B with R rotating weight copies."""

    def __init__(self, name, shapes, B, seed=0, min_rotation_bytes=3 * L2_BYTES, layers=1,
                 extra=None, fused=None):
        import torch
        import gemm_zq_rmsnorm_gb300 as zq
        self.zq, self.torch = zq, torch
        self.name, self.B = name, B
        # B = 1: one launch per layer input normalises it and runs every
        # projection that reads it (zq_rmsnorm_q4k_gemv); otherwise
        # RMSNorm+Q8_1 first, then one call per projection
        self.fused = (B == 1) if fused is None else fused
        self.prefetch = False   # fused launches pulling the next launch's weights into L2 (--l2-prefetch)
        dev = "cuda"
        self.extra = list(extra or [])
        self.shapes = shapes + self.extra
        # distinct inputs per projection input width; the norm runs once per
        # distinct input (q/k/v share the attention input, gate/up the FFN one)
        self.inputs_K = layer_inputs(shapes)
        self.x = {k: torch.from_numpy(inputs.activations(seed + i, B, K)).to(dev)
                  for i, (k, K) in enumerate(self.inputs_K)}
        self.g = {k: torch.from_numpy(inputs.gamma(seed + i, K)).to(dev)
                  for i, (k, K) in enumerate(self.inputs_K)}
        self.a = {k: zq.empty_q8_1(B, K, dev) for k, K in self.inputs_K}
        # weights: generate once per shape, clone to distinct device copies
        self.layer_shapes = list(shapes)
        self.R = rotation_copies(self.layer_shapes, layers, self.extra, min_rotation_bytes)
        self.layers = layers
        base = {}
        for si, (pname, K, N, paired) in enumerate(self.shapes):
            w1 = torch.from_numpy(inputs.q4k_weights(seed + 17 * si, N, K)).to(dev)
            w2 = torch.from_numpy(inputs.q4k_weights(seed + 17 * si, N, K, tag_offset=100)).to(dev) if paired else None
            base[pname] = (w1, w2)

        def clone(names):
            return {k: (base[k][0].clone(), None if base[k][1] is None else base[k][1].clone()) for k in names}

        lnames = [p for (p, _, _, _) in self.layer_shapes]
        enames = [p for (p, _, _, _) in self.extra]
        # W[copy] = (list over layers of {name: (W, W2)}, {extra name: (W, W2)})
        self.W = []
        for r in range(self.R):
            layers_w = [({k: base[k] for k in lnames} if (r == 0 and li == 0) else clone(lnames))
                        for li in range(layers)]
            extra_w = {k: base[k] for k in enames} if r == 0 else clone(enames)
            self.W.append((layers_w, extra_w))
        self.y = {}
        for (pname, K, N, paired) in self.shapes:
            self.y[pname] = (torch.empty((B, N), dtype=torch.float32, device=dev),
                             torch.empty((B, N), dtype=torch.float32, device=dev) if paired else None)
        self.key_of = {p: input_key(p) for (p, _, _, _) in self.layer_shapes}
        for (p, K, N, _) in self.extra:
            self.key_of[p] = [k for k, KK in self.inputs_K if KK == K][0]
        # B > 1: the matrices of a layer that read the same input are stored
        # row-stacked as one Q4_K matrix ([Wq; Wk; Wv], [Wgate; Wup]: the same
        # bytes, one activation split and one launch per input)
        self.stacked = B > 1 and not self.fused
        self.groups = []   # (input key, K, N_total)
        if self.stacked:
            for k, K in self.inputs_K:
                n_tot = sum(N * (2 if p else 1) for (pn, KK, N, p) in self.layer_shapes if self.key_of[pn] == k)
                if n_tot:
                    self.groups.append((k, K, n_tot))
            self.SW = []   # SW[copy][layer][input key]
            for r in range(self.R):
                layers_w, _ = self.W[r]
                per_layer = []
                for li in range(layers):
                    d = {}
                    for k, K, _ in self.groups:
                        parts = []
                        for (pn, KK, N, p) in self.layer_shapes:
                            if self.key_of[pn] == k:
                                parts += [w for w in layers_w[li][pn] if w is not None]
                        d[k] = torch.cat(parts)
                    per_layer.append(d)
                self.SW.append(per_layer)
            self.gy = {k: torch.empty((B, n), dtype=torch.float32, device=dev) for k, _, n in self.groups}
        ws = max(zq.gemm_workspace_bytes(N, K, B) for (_, K, N, _) in self.shapes)
        if self.stacked:
            ws = max([ws] + [zq.gemm_workspace_bytes(n, K, B) for _, K, n in self.groups])
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def weights(self, r, pname, layer=0):
        layers_w, extra_w = self.W[r]
        return extra_w[pname] if pname in extra_w else layers_w[layer][pname]

    def _proj(self, pname, K, N, paired, w1, w2, stream):
        zq = self.zq
        a = self.a[self.key_of[pname]]
        y1, y2 = self.y[pname]
        if self.B == 1:
            if paired:
                zq.q4k_gemv_pair(w1, w2, N, K, a, y1, y2, stream=stream)
            else:
                zq.q4k_gemv(w1, N, K, a, y1, stream=stream)
        else:
            zq.q4k_gemm(w1, N, K, a, self.B, y1, self.ws, stream=stream)
            if paired:
                zq.q4k_gemm(w2, N, K, a, self.B, y2, self.ws, stream=stream)

    def fused_groups(self, r, layer=0):
        """(input key, K, [W], [N], [y]) per fused launch: the matrices of one
        layer that read the same input, at most four per launch."""
        layers_w, extra_w = self.W[r]
        out = []
        for k, K in self.inputs_K:
            mats = []
            for (pname, KK, N, paired) in self.layer_shapes:
                if self.key_of[pname] != k:
                    continue
                w1, w2 = layers_w[layer][pname]
                y1, y2 = self.y[pname]
                mats.append((w1, N, y1[0]))
                if paired:
                    mats.append((w2, N, y2[0]))
            for i in range(0, len(mats), 4):
                c = mats[i:i + 4]
                out.append((k, K, [m[0] for m in c], [m[1] for m in c], [m[2] for m in c]))
        return out

    def _fused_calls(self, r):
        calls = []
        for li in range(self.layers):
            calls += self.fused_groups(r, li)
        layers_w, extra_w = self.W[r]
        for (pname, K, N, paired) in self.extra:
            w1, w2 = extra_w[pname]
            y1, y2 = self.y[pname]
            Ws, Ns, ys = [w1], [N], [y1[0]]
            if paired:
                Ws, Ns, ys = Ws + [w2], Ns + [N], ys + [y2[0]]
            calls.append((self.key_of[pname], K, Ws, Ns, ys))
        return calls

    # bytes of the next launch's first matrix that a fused launch pulls into L2
    PREFETCH_MAX = 32 << 20

    def _run_fused(self, r, stream):
        zq = self.zq
        calls = self._fused_calls(r)
        after = self._fused_calls((r + 1) % self.R)[0]   # the next step starts on the next copy
        for i, (k, K, Ws, Ns, ys) in enumerate(calls):
            nxt = calls[i + 1] if i + 1 < len(calls) else after
            pf = nxt[2][0] if self.prefetch else None
            zq.rmsnorm_q4k_gemv(self.x[k][0], self.g[k], inputs.EPS, Ws, Ns, ys, stream=stream, l2_prefetch=pf,
                                l2_prefetch_bytes=min(pf.numel(), self.PREFETCH_MAX) if pf is not None else 0)

    # one pass of the path
    def run(self, r=0, stream=None):
        if self.fused:
            return self._run_fused(r, stream)
        layers_w, extra_w = self.W[r]
        if self.stacked:
            # one call per input: RMSNorm + Q8_1 (and, for B >= 5, the
            # activation split) in one kernel, then the projection
            for li in range(self.layers):
                for k, K, n in self.groups:
                    # the codes themselves are needed only by the streamed path (B <= 4)
                    self.zq.rmsnorm_q4k_gemm(self.x[k], self.g[k], inputs.EPS, self.SW[r][li][k], n, y=self.gy[k],
                                             q8_out=self.a[k] if self.B <= 4 else None, workspace=self.ws,
                                             stream=stream)
            for (pname, K, N, paired) in self.extra:
                w1, w2 = extra_w[pname]
                self._proj(pname, K, N, paired, w1, w2, stream)
            return
        for k, K in self.inputs_K:
            self.zq.rmsnorm_q8_1(self.x[k], self.g[k], inputs.EPS, out=self.a[k], stream=stream)
        for li in range(self.layers):
            for (pname, K, N, paired) in self.layer_shapes:
                w1, w2 = layers_w[li][pname]
                self._proj(pname, K, N, paired, w1, w2, stream)
        for (pname, K, N, paired) in self.extra:
            w1, w2 = extra_w[pname]
            self._proj(pname, K, N, paired, w1, w2, stream)

    def launches_per_step(self):
        if self.fused:
            return len(self.fused_groups(0)) * self.layers + len(self.extra)
        n = 0 if self.stacked else len(self.inputs_K)
        if self.stacked:
            calls = [(K, N, False) for _, K, N in self.groups] * self.layers + \
                    [(K, N, p) for (_, K, N, p) in self.extra]
        else:
            calls = [(K, N, p) for (_, K, N, p) in self.layer_shapes * self.layers + self.extra]
        for (K, N, paired) in calls:
            calls = 1 if (self.B == 1 or not paired) else 2
            if self.B == 1:
                per = 1
            elif self.B <= 4:
                per = 2 if self.stacked else 1   # (norm +) the streamed mat-vec with the tokens staged together
            else:
                # q8 split + GEMM, + the split-K reduction when the workspace
                # holds partial sums beyond the hi/lo activations and scales
                pad = lambda n: (n + 255) // 256 * 256
                base = 4 * self.B * K + pad(4 * self.B) + pad(self.B * K // 8)
                # (stacked: the norm writes the split) + GEMM + reduction or fixup
                per = 2 + (1 if self.zq.gemm_workspace_bytes(N, K, self.B) > base else 0)
            n += calls * per
        return n

    def algo_bytes(self):
        return layer_algo_bytes(self.layer_shapes, self.B, self.layers, self.extra)

    def algo_ops(self):
        return sum(2 * self.B * N * K * (2 if p else 1) for (_, K, N, p) in self.layer_shapes * self.layers + self.extra)

    def input_bytes(self):
        return sum(self.B * K * 4 for _, K in self.inputs_K)

    def output_bytes(self):
        return sum(self.B * N * 4 * (2 if p else 1) for (_, K, N, p) in self.shapes)


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
                for nm, v in zip(names, r[3:7]):
                    if v.lower() == "active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def time_graphs(torch, graphs, steps, warmup, stream):
    """Replay graphs round-robin; W untimed, K timed; returns ms per step."""
    for i in range(warmup):
        graphs[i % len(graphs)].replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def capture(torch, fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # uncaptured call first: sets per-device kernel attributes
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def time_steps(torch, run, R, steps, warmup, stream):
    """ms per step over exactly `steps` timed steps (after at least `warmup`
    untimed ones), step i on weight copy i % R.  Consecutive steps are
    captured together, S = R * ceil(8 / R) of them per CUDA graph (a whole
    number of passes over the copies), so they run without a graph-launch
    gap between them, as a forward pass captured once would; a remainder
    graph makes the count exact.  Each step is still a full pass of the
    path over its own weight copy."""
    S = R * max(1, -(-8 // R))
    full = capture(torch, lambda: [run(i % R) for i in range(S)], stream)
    tail_n = steps % S
    tail = capture(torch, lambda: [run(i % R) for i in range(tail_n)], stream) if tail_n else None
    for _ in range(max(1, -(-warmup // S))):
        full.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps // S):
            full.replay()
        if tail is not None:
            tail.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def bench_workload(torch, wl, steps, warmup, stream):
    if wl.B == 1:
        # decode: several consecutive steps per graph
        return time_steps(torch, wl.run, wl.R, steps, warmup, stream), None
    # batched steps (each several hundred microseconds to a millisecond):
    # one graph per step
    graphs = [capture(torch, lambda r=r: wl.run(r), stream) for r in range(wl.R)]
    ms = time_graphs(torch, graphs, steps, warmup, stream)
    return ms, graphs


def bench_dominant(torch, wl, pname, steps, warmup, stream):
    """Average duration of the workload's largest kernel alone (CUDA events
    around back-to-back launches on its stream, rotating weight copies)."""
    (_, K, N, paired) = [s for s in wl.shapes if s[0] == pname][0]
    zq = wl.zq
    a = wl.a[wl.key_of[pname]]
    if wl.stacked:
        # the launch of the row-stacked matrix holding this projection
        key = wl.key_of[pname]
        (_, K, N) = [g for g in wl.groups if g[0] == key][0]
        g = capture(torch, lambda: [zq.q4k_gemm(wl.SW[i % wl.R][0][key], N, K, a, wl.B, wl.gy[key], wl.ws)
                                    for i in range(4 * wl.R)], stream)
        ms = time_graphs(torch, [g], max(3, steps // 4), max(1, warmup // 2), stream) / (4 * wl.R)
        alg = proj_bytes(K, N, wl.B) if wl.B <= 16 else 2 * wl.B * N * K
        return ms, alg, (K, N, False)

    def one(r):
        w1, w2 = wl.weights(r, pname)
        y1, y2 = wl.y[pname]
        if wl.fused:
            k = wl.key_of[pname]
            Ws, Ns, ys = ([w1, w2], [N, N], [y1[0], y2[0]]) if paired else ([w1], [N], [y1[0]])
            zq.rmsnorm_q4k_gemv(wl.x[k][0], wl.g[k], inputs.EPS, Ws, Ns, ys)
        elif wl.B == 1:
            if paired:
                zq.q4k_gemv_pair(w1, w2, N, K, a, y1, y2)
            else:
                zq.q4k_gemv(w1, N, K, a, y1)
        else:
            zq.q4k_gemm(w1, N, K, a, wl.B, y1, wl.ws)

    # one graph holds several launches (rotating weight copies), so the timing
    # is the kernel's device time, not the host's per-replay overhead
    per_graph = 4 * wl.R
    g = capture(torch, lambda: [one(i % wl.R) for i in range(per_graph)], stream)
    reps = max(3, steps // 4)
    ms = time_graphs(torch, [g], reps, max(1, warmup // 2), stream) / per_graph
    units = 2 if (paired and wl.B == 1) else 1
    if wl.fused:
        # weights once, x and gamma (the kernel normalises and packs x itself), y
        alg = units * N * K * 144 // 256 + 2 * K * 4 + units * N * 4
    elif wl.B == 1:
        alg = proj_bytes(K, N, 1) * units - (K * (1 + 4 / 32) if units == 2 else 0)
    elif wl.B <= 4:
        alg = proj_bytes(K, N, wl.B)     # streamed: weights once for the B tokens
    else:
        alg = 2 * wl.B * N * K
    return ms, alg, (K, N, paired)


def silu_down(torch, wl, steps, warmup, stream):
    """The FFN down projection fed by SiLU(gate) * up of the layer's gate/up
    outputs: Q8_1 packing inside the mat-vec launch (zq_silu_q4k_gemv) against
    a separate packing launch (zq_silu_mul_q8_1) followed by zq_q4k_gemv.
    Per-launch device times over graphs of back-to-back calls, rotating
    weight copies."""
    zq = wl.zq
    (_, K, N, _) = [sh for sh in wl.shapes if sh[0] == "down"][0]
    yg, yu = wl.y["gate_up"]
    g, u = yg[0], yu[0]
    y = wl.y["down"][0]
    a = zq.empty_q8_1(1, K)
    per = 4 * wl.R

    def fused():
        for i in range(per):
            zq.silu_q4k_gemv(g, u, [wl.weights(i % wl.R, "down")[0]], [N], [y[0]])

    def two_step():
        for i in range(per):
            zq.silu_mul_q8_1(yg, yu, out=a)
            zq.q4k_gemv(wl.weights(i % wl.R, "down")[0], N, K, a, y[0])

    reps = max(3, steps // 4)
    tf = time_graphs(torch, [capture(torch, fused, stream)], reps, max(1, warmup // 2), stream) / per
    tt = time_graphs(torch, [capture(torch, two_step, stream)], reps, max(1, warmup // 2), stream) / per
    return {"projection": f"down {K}->{N} fed by silu(gate)*up", "fused_us": round(tf * 1e3, 2),
            "two_step_us": round(tt * 1e3, 2), "fused_gain": round(tt / tf, 3),
            "fused_gbs": round(N * K * 144 / 256 / (tf * 1e-3) / 1e9, 1)}


def dequant_then_gemm(torch, wl, steps, warmup, stream):
    """The dequantise-then-GEMM design measured beside the library's own
    prefill, all in the library's kernels (no library GEMM): every
    projection's Q4_K weights dequantised to binary16 (zq_q4k_dequant_f16),
    the Q8_1 activations to binary16 q8*d8 (zq_q8_1_dequant_f16), then the
    tcgen05 binary16 GEMM (zq_f16_gemm).  Its error is reported against the
    library's exact-product path on the gate projection, with
    S = sum |x16 * w16| from the same GEMM on magnitudes."""
    zq = wl.zq
    B = wl.B
    maxNK = max(N * K for (_, K, N, _) in wl.shapes)
    wbuf = torch.empty(maxNK, dtype=torch.float16, device="cuda")
    x16 = {k: torch.empty((B, K), dtype=torch.float16, device="cuda") for k, K in wl.inputs_K}
    ymax = max(N for (_, _, N, _) in wl.shapes)
    ybuf = torch.empty(B * ymax, dtype=torch.float32, device="cuda")
    wsb = max(zq.f16_gemm_workspace_bytes(N, K, B) for (_, K, N, _) in wl.shapes)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")

    def step(r, only=None):
        for k, K in wl.inputs_K:
            zq.rmsnorm_q8_1(wl.x[k], wl.g[k], inputs.EPS, out=wl.a[k], stream=stream)
            zq.q8_1_dequant_f16(wl.a[k], out=x16[k], stream=stream)
        layers_w, _ = wl.W[r]
        for (pname, K, N, paired) in wl.layer_shapes:
            if only and pname != only:
                continue
            for w in layers_w[0][pname]:
                if w is None:
                    continue
                wd = zq.q4k_dequant_f16(w, N, K, out=wbuf[:N * K].view(N, K), stream=stream)
                zq.f16_gemm(wd, N, K, x16[wl.key_of[pname]], B, y=ybuf[:B * N].view(B, N), workspace=ws,
                            stream=stream)

    graphs = [capture(torch, lambda r=r: step(r), stream) for r in range(wl.R)]
    with Clocks(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ms = time_graphs(torch, graphs, steps, warmup, stream)
    # the gate projection alone: dequantisation, then the GEMM
    (_, K, N, _) = [sh for sh in wl.shapes if sh[0] == "gate_up"][0]
    xg = x16[wl.key_of["gate_up"]]
    wd = wbuf[:N * K].view(N, K)
    yg = ybuf[:B * N].view(B, N)
    gd = capture(torch, lambda: [zq.q4k_dequant_f16(wl.weights(i % wl.R, "gate_up")[0], N, K, out=wd,
                                                    stream=stream) for i in range(4)], stream)
    gm = capture(torch, lambda: [zq.f16_gemm(wd, N, K, xg, B, y=yg, workspace=ws, stream=stream)
                                 for _ in range(4)], stream)
    d_ms = time_graphs(torch, [gd], max(3, steps // 4), 2, stream) / 4
    m_ms = time_graphs(torch, [gm], max(3, steps // 4), 2, stream) / 4
    # error of the design on the gate projection: against the library's
    # exact-product path (itself within 1e-4 * S of the oracle)
    w0 = wl.weights(0, "gate_up")[0]
    with torch.cuda.stream(stream):
        zq.q4k_dequant_f16(w0, N, K, out=wd, stream=stream)
        y_dq = zq.f16_gemm(wd, N, K, xg, B, workspace=ws, stream=stream)
        S16 = zq.f16_gemm(wd.abs(), N, K, xg.abs(), B, workspace=ws, stream=stream)
        y_ex = zq.q4k_gemm(w0, N, K, wl.a[wl.key_of["gate_up"]], B, stream=stream)
    torch.cuda.synchronize()
    rel = ((y_dq.double() - y_ex.double()).abs() / S16.double().clamp_min(1e-30)).max().item()
    gate_flops = 2 * B * N * K
    del wbuf, ybuf, ws
    return {"design": "dequantise-then-GEMM, all in-library: zq_q4k_dequant_f16 + zq_q8_1_dequant_f16 + "
                      "zq_f16_gemm (tcgen05 kind::f16, CTA pairs); no library GEMM",
            "ms_per_step": round(ms, 4), "value": round(wl.algo_ops() / (ms * 1e-3) / 1e12, 2), "unit": "TOPS",
            "gate_dequant_ms": round(d_ms, 5), "gate_gemm_ms": round(m_ms, 5),
            "gate_gemm_tflops": round(gate_flops / (m_ms * 1e-3) / 1e12, 1),
            "max_err_over_S_vs_exact_path": float(f"{rel:.3e}"),
            "clocks": clk.summary(),
            "note": "binary16 weights and activations: each product carries the two binary16 roundings "
                    "(about 2^-10 * S at worst), unlike the library's exact hi/lo products; the dequantised "
                    "weight copy is 3.6x the Q4_K bytes"}


# Q5_K / Q6_K rows: the LM head of the small model in Q6_K (with and without
# the final RMSNorm fused in) and the recurrent output projection of the
# 27B-class layer (value width 48 x 128 = 6144 -> hidden 5120) in Q5_K.
KQUANT_CASES = [  # (label, fmt, K, N, B, fused)
    ("q6k_lm_head", "q6k", 1024, 151936, 1, False),
    ("q6k_lm_head_fused_norm", "q6k", 1024, 151936, 1, True),
    ("q5k_recurrent_out", "q5k", 6144, 5120, 1, False),
    ("q5k_recurrent_out_b4", "q5k", 6144, 5120, 4, False),
]
KQ_BLOCK = {"q5k": 176, "q6k": 210}


def kquant_rows(torch, steps, warmup, stream, pk):
    """Per-launch device time of each Q5_K / Q6_K case over graphs of
    back-to-back launches on rotating weight copies (>= 3x L2), as algorithmic
    HBM GB/s: weights once + activations (Q8_1 codes, or x and gamma when the
    norm is fused) + y."""
    import gemm_zq_rmsnorm_gb300 as zq
    out = []
    for (label, fmt, K, N, B, fused) in KQUANT_CASES:
        wbytes = N * K // 256 * KQ_BLOCK[fmt]
        R = max(2, -(-3 * L2_BYTES // wbytes))
        gen = inputs.q5k_weights if fmt == "q5k" else inputs.q6k_weights
        w0 = torch.from_numpy(gen(0, N, K)).cuda()
        Ws = [w0] + [w0.clone() for _ in range(R - 1)]
        x = torch.from_numpy(inputs.activations(1, B, K)).cuda()
        g = torch.from_numpy(inputs.gamma(1, K)).cuda()
        a = zq.rmsnorm_q8_1(x, g, inputs.EPS)
        y = torch.empty((B, N), dtype=torch.float32, device="cuda")
        per = 2 * R

        def calls():
            for i in range(per):
                if fused:
                    zq.rmsnorm_q6k_gemv(x[0], g, inputs.EPS, Ws[i % R], N, y=y[0])
                else:
                    zq.kq_gemm(fmt, Ws[i % R], N, K, a, B, y=y)

        calls()
        torch.cuda.synchronize()
        reps = max(3, steps // 4)
        ms = time_graphs(torch, [capture(torch, calls, stream)], reps, max(2, warmup // 2), stream)
        ms /= per
        act = 2 * K * 4 if fused else B * K * (1 + 4 / 32)
        alg = wbytes + act + B * N * 4
        launches = 1 if B == 1 else -(-B // 4)
        gbs = alg / (ms * 1e-3) / 1e9
        out.append({"case": label, "format": fmt.upper().replace("K", "_K"), "K": K, "N": N, "B": B,
                    "call": ("zq_rmsnorm_q6k_gemv" if fused else f"zq_{fmt}_{'gemv' if B == 1 else 'gemm'}"),
                    "launches": launches, "us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                    "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4), "weight_copies_rotated": R,
                    "timed_launches": reps * per * launches})
        del Ws, w0
        torch.cuda.empty_cache()
    return out


_ORACLE_CACHE = {}


def oracle_sample(wl_shapes, B, budget_s=12.0, seed=0):
    """Time the CPU oracle on a bounded sample: RMSNorm+Q8_1 of every input and
    a row sample of every projection; returns (seconds per full step, sample text)."""
    import oracle
    t_total, frac_used = 0.0, []
    seen = {}
    per_shape_budget = budget_s / max(1, len(wl_shapes))
    for si, (pname, K, N, paired) in enumerate(wl_shapes):
        key = input_key(pname)
        if key not in seen:
            x = inputs.activations(seed + si, B, K)
            g = inputs.gamma(seed + si, K)
            t0 = time.perf_counter()
            q = oracle.rmsnorm_q8_1(x, g, inputs.EPS)
            t_total += time.perf_counter() - t0
            seen[key] = q
        qs, d, s = seen[key]
        ck = (seed + 17 * si, N, K)
        if ck not in _ORACLE_CACHE:
            _ORACLE_CACHE[ck] = inputs.q4k_weights(seed + 17 * si, N, K)
        W = _ORACLE_CACHE[ck]
        # calibrate on a few rows, then take as many as fit the budget
        rows = np.arange(min(N, 8), dtype=np.int32)
        t0 = time.perf_counter()
        oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows, want_scale=False)
        dt = max(time.perf_counter() - t0, 1e-6) / len(rows)
        n_rows = int(min(N, max(8, per_shape_budget / dt / (2 if paired else 1))))
        rows = np.linspace(0, N - 1, n_rows).astype(np.int32)
        t0 = time.perf_counter()
        oracle.q4k_matmul(W, N, K, qs, d, s, rows=rows, want_scale=False)
        dt = time.perf_counter() - t0
        t_total += dt * (N / n_rows) * (2 if paired else 1)
        frac_used.append(f"{pname} {n_rows}/{N} rows")
    return t_total, "; ".join(frac_used)


# ----------------------------------------------------------------------------
def reduce_max_over_ranks(dist, v, device):
    """The slowest rank's time: max of v over the process group (v itself
    without one)."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms_max, world):
    """Replicas: every rank processes the same units; the job's rate is all
    ranks' units over the slowest rank's time (units per second)."""
    return units_per_rank * world / (ms_max * 1e-3)


def decode_record(torch, wl, steps, warmup, stream, pk, local_rank, max_over_ranks, world, barrier):
    """One B = 1 decode workload: the step's rate in HBM GB/s of algorithmic
    bytes, its dominant launch against the HBM roofline, clocks."""
    barrier()
    with Clocks(local_rank) as clk:
        ms, _ = bench_workload(torch, wl, steps, warmup, stream)
    ms = max_over_ranks(ms)
    gbs = whole_job_rate(wl.algo_bytes(), ms, world) / 1e9
    # the dominant launch: the one moving the most weight bytes
    dom = max(wl.shapes, key=lambda s: s[1] * s[2] * (2 if s[3] else 1))[0]
    dms, dalg, (dK, dN, dp) = bench_dominant(torch, wl, dom, steps, warmup, stream)
    achieved = dalg / (dms * 1e-3) / 1e9
    return {
        "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(ms, 5),
        "config": decode_config(wl.name, wl.layer_shapes, wl.layers, wl.extra, wl.R, wl.fused, wl.prefetch),
        "roofline": {"bound": "hbm",
                     "kernel": (f"rmsnorm_q4k_gemv {dK}->{dN}{' x2 (gate+up)' if dp else ''}" if wl.fused
                                else f"q4k_gemv{'_pair' if dp else ''} {dK}->{dN}"),
                     "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / pk["hbm_gbs"], 4), "peak_source": pk["source"] + " (burst copy)",
                     "traffic": (recorded_traffic(f"{'fused_' if wl.fused else ''}q4k_gemv_stream_pair_{dK}x{dN}")
                                 if dp else None),
                     "kernel_ms": round(dms, 5)},
        "gpu_launches": wl.launches_per_step() * steps,
        "clocks": clk.summary(),
    }


def batch_record(torch, B, shapes, name, steps, warmup, stream, pk, local_rank, max_over_ranks, world, barrier,
                 compare_dequant=False):
    """One batched workload (B tokens through every projection): effective
    TOPS and HBM GB/s of the step; the dominant projection against the HBM
    roofline (B <= 16: weights read once for all tokens) or the tensor
    roofline (B > 16)."""
    wl = LayerWorkload(name, shapes, B)
    barrier()
    with Clocks(local_rank) as clk:
        ms, _ = bench_workload(torch, wl, steps, warmup, stream)
    ms = max_over_ranks(ms)
    tops = whole_job_rate(wl.algo_ops(), ms, world) / 1e12
    gbs = whole_job_rate(wl.algo_bytes(), ms, world) / 1e9
    dom = "gate_up" if any(s[0] == "gate_up" for s in wl.shapes) else wl.shapes[0][0]
    dms, dalg, (dK, dN, dp) = bench_dominant(torch, wl, dom, steps, warmup, stream)
    if B <= 16:
        (_, _, N, _) = [s for s in wl.shapes if s[0] == dom][0]
        alg_bytes = proj_bytes(dK, dN, B)
        ach = alg_bytes / (dms * 1e-3) / 1e9
        path = "streamed mat-vec, tokens staged together" if B <= 4 else "chunk kernel on CTA pairs"
        roof = {"bound": "hbm", "kernel": f"q4k_gemm {dK}->{dN} B={B} ({path})",
                "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / pk["hbm_gbs"], 4), "peak_source": pk["source"] + " (burst copy)",
                "traffic": recorded_traffic(f"q4k_gemm_chunk_{B}x{dK}x{dN}"), "kernel_ms": round(dms, 5),
                "algorithmic_bytes_per_launch": int(alg_bytes)}
    else:
        ach = dalg / (dms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": f"q4k_gemm {dK}->{dN} B={B}",
                "achieved": round(ach, 2), "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops"], 4),
                "peak_source": pk["source"] + " bf16 dense burst (fp16 operands run at the bf16 rate; "
                               "int8 tcgen05 is not available on sm_103a)",
                "traffic": recorded_traffic(f"q4k_gemm_tc_{B}x{dK}x{dN}"),
                "kernel_ms": round(dms, 5)}
    rec = {"workload": wl.name, "B": B, "value": round(tops, 2), "unit": "TOPS",
           "ms_per_step": round(ms, 4), "hbm_gbs": round(gbs, 1),
           "weights": "row-stacked per input: [q;k;v] (5120 -> 8192), o, [gate;up] (5120 -> 34816), down; "
                      "one activation split and one launch per input",
           "algorithmic_ops_per_step": int(wl.algo_ops()), "algorithmic_bytes_per_step": int(wl.algo_bytes()),
           "roofline": roof,
           "gpu_launches": wl.launches_per_step() * steps, "clocks": clk.summary()}
    if compare_dequant:
        rec["dequant_then_gemm"] = dequant_then_gemm(torch, wl, steps, warmup, stream)
    del wl
    torch.cuda.empty_cache()
    return rec


def peak_probes(torch, stream, local_rank, sms):
    """Throughput of the arithmetic the projection kernels can use (in-library
    probes, zq_debug_peak_probe): packed int8 dot products (dp4a), the legacy
    warp-level int8 MMA (mma.sync m16n8k32 s8) and the tcgen05 binary16 MMA
    (kind::f16, 128 x 256 x 16, one issuing thread per SM).  Each probe is
    one launch of about a millisecond, timed with CUDA events after one
    warm-up launch."""
    import gemm_zq_rmsnorm_gb300 as zq
    out = {}
    sink = torch.empty(sms * 8 * 256, dtype=torch.int32, device="cuda")
    cfg = {0: (sms * 8, 40000), 1: (sms * 8, 6000), 2: (sms, 40000), 3: (sms, 40000), 4: (sms, 40000),
           5: (sms, 40000), 6: (sms, 40000), 7: (sms, 40000), 8: (sms, 40000), 9: (sms, 40000), 10: (sms, 40000)}
    with Clocks(local_rank) as clk:
        for kind, (blocks, iters) in cfg.items():
            with torch.cuda.stream(stream):
                zq.debug_peak_probe(kind, blocks, max(1, iters // 8), sink, stream=stream)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                zq.debug_peak_probe(kind, blocks, iters, sink, stream=stream)
                e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            ops = zq.probe_ops(kind, blocks, iters)
            out[zq.PROBE_KINDS[kind]] = {"tera_ops_per_s": round(ops / (ms * 1e-3) / 1e12, 1), "ms": round(ms, 4),
                                         "ops": ops, "blocks": blocks}
            if kind >= 2:   # one issuing thread per SM: time per MMA instruction
                out[zq.PROBE_KINDS[kind]]["ns_per_mma"] = round(ms * 1e6 / iters, 2)
    assert zq.device_status() == 0, "a probe's bounded wait expired"
    out["clocks"] = clk.summary()
    out["note"] = ("tcgen05.mma kind::i8 is rejected by ptxas for sm_103a, so the prefill path runs binary16 MMAs on "
                   "exact hi/lo halves of every Q8_1 value (two MMAs per K step); its effective int8-op rate is "
                   "compared with these measured rates")
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="zq", choices=["zq", "reference"])
    ap.add_argument("--workload", default="headline",
                    choices=["headline", "decode-27b", "decode-small", "chunk", "prefill-512", "tiny", "kquants",
                             "peaks"])
    ap.add_argument("--chunk-batch", type=int, default=0,
                    help="--workload chunk: run only this chunk size (one of %s)" % (inputs.CHUNK_BATCHES,))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--l2-prefetch", action="store_true",
                    help="fused decode launches pull the next launch's weights into L2 (measured slower on this kernel)")
    ap.add_argument("--no-l2-prefetch", action="store_true", help="the default; kept for older command lines")
    ap.add_argument("--no-compare-dequant", action="store_true",
                    help="skip the dequantise-then-GEMM comparison on the 512-token layer")
    ap.add_argument("--compare-dequant", action="store_true", help="the default; kept for older command lines")
    ap.add_argument("--decode-path", default="fused", choices=["fused", "two-step"],
                    help="B = 1 step: fused RMSNorm+mat-vec launches, or RMSNorm+Q8_1 then per-projection calls")
    args = ap.parse_args()
    assert args.warmup >= 3 or args.impl == "reference" or os.environ.get("ZQ_BENCH_DEBUG"), "W >= 3"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args)

    import torch
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    stream = torch.cuda.Stream()
    pk = peaks()
    sms = torch.cuda.get_device_properties(local_rank).multi_processor_count
    out = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic"}

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return reduce_max_over_ranks(dist, v, "cuda")

    common = dict(stream=stream, pk=pk, local_rank=local_rank, max_over_ranks=max_over_ranks, world=world,
                  barrier=barrier)
    fz = args.decode_path == "fused"
    # the secondary workloads run with fewer timed steps: the line must finish in minutes
    sub_steps = max(3, args.steps // 4)

    def decode_wl(which):
        if which == "decode-27b":
            wl = LayerWorkload("decode-27b-layer", inputs.LAYER_27B, 1, fused=fz)
        elif which == "decode-small":
            wl = LayerWorkload("decode-small-28L+lm_head", inputs.SMALL_DECODE[:-1], 1, layers=28,
                               extra=[inputs.SMALL_DECODE[-1]], fused=fz)
        else:
            wl = LayerWorkload("tiny-1024x1024", inputs.TINY, 1, min_rotation_bytes=3 * L2_BYTES, fused=fz)
        wl.prefetch = args.l2_prefetch and not args.no_l2_prefetch
        return wl

    if args.workload in ("headline", "decode-27b", "decode-small", "tiny"):
        which = "decode-27b" if args.workload == "headline" else args.workload
        wl_dec = decode_wl(which)
        rec = decode_record(torch, wl_dec, args.steps, args.warmup, **common)
        out.update(rec)
        out["dtype"] = "u8"
        if any(sh[0] == "down" for sh in wl_dec.shapes) and any(sh[0] == "gate_up" for sh in wl_dec.shapes):
            out["silu_down"] = silu_down(torch, wl_dec, args.steps, args.warmup, stream)
        if not args.no_e2e:
            out["e2e"] = e2e(torch, wl_dec, args.steps, args.warmup)
        if rank == 0 and not args.no_cpu_baseline:
            secs, sample = oracle_sample(wl_dec.shapes, 1, budget_s=10.0)
            out["cpu_baseline"] = {"value": round(wl_dec.algo_bytes() / secs / 1e9, 4), "unit": "GB/s",
                                   "cores": 1, "kind": "oracle",
                                   "sample": f"RMSNorm+Q8_1 of every input, row samples: {sample}; "
                                             f"scaled to one full step ({secs:.2f} s per step)"}
        del wl_dec
        torch.cuda.empty_cache()
        if args.workload == "headline":
            # the other configurations of the same path, each with its own
            # roofline and clocks
            for key, which in (("small_model_28L", "decode-small"), ("tiny", "tiny")):
                wl = decode_wl(which)
                out[key] = decode_record(torch, wl, sub_steps, args.warmup, **common)
                del wl
                torch.cuda.empty_cache()

    if args.workload in ("headline", "prefill-512"):
        rec = batch_record(torch, inputs.PREFILL_B, inputs.LAYER_27B, f"prefill-{inputs.PREFILL_B}",
                           max(3, args.steps // 5), args.warmup, compare_dequant=not args.no_compare_dequant,
                           **common)
        if args.workload == "prefill-512":
            out.update({"value": rec["value"], "unit": "TOPS", "ms_per_step": rec["ms_per_step"], "dtype": "u8",
                        "config": {"workload": rec["workload"], "B": rec["B"]}, "roofline": rec["roofline"],
                        "gpu_launches": rec["gpu_launches"], "clocks": rec["clocks"]})
            if "dequant_then_gemm" in rec:
                out["dequant_then_gemm"] = rec["dequant_then_gemm"]
        else:
            if "dequant_then_gemm" in rec:
                out["dequant_then_gemm"] = rec.pop("dequant_then_gemm")
            out["prefill_b512"] = rec

    if args.workload in ("headline", "chunk"):
        batches = [b for b in inputs.CHUNK_BATCHES if args.workload == "headline" or not args.chunk_batch
                   or b == args.chunk_batch]
        recs = [batch_record(torch, B, inputs.CHUNK_SHAPES, f"chunk-B{B}", sub_steps, args.warmup, **common)
                for B in batches]
        if args.workload == "chunk":
            r0 = recs[0]
            out.update({"value": r0["hbm_gbs"], "unit": "GB/s", "ms_per_step": r0["ms_per_step"], "dtype": "u8",
                        "config": {"workload": r0["workload"], "B": r0["B"]}, "roofline": r0["roofline"],
                        "gpu_launches": r0["gpu_launches"], "clocks": r0["clocks"], "more": recs[1:]})
        else:
            out["chunk"] = {f"B{r['B']}": r for r in recs}

    if args.workload in ("headline", "kquants"):
        barrier()
        with Clocks(local_rank) as clk:
            kq = kquant_rows(torch, sub_steps if args.workload == "headline" else args.steps, args.warmup, stream, pk)
        if args.workload == "kquants":
            r0 = kq[0]
            out.update({"value": r0["gbs"], "unit": "GB/s", "ms_per_step": round(r0["us"] / 1e3, 5), "dtype": "u8",
                        "config": {"workload": f"{r0['case']} {r0['K']}->{r0['N']} B={r0['B']}",
                                   "l2": "inputs larger than L2: rotating weight copies"},
                        "roofline": {"bound": "hbm", "kernel": f"{r0['call']} {r0['K']}->{r0['N']}",
                                     "achieved": r0["gbs"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                                     "frac": r0["frac_of_hbm"], "peak_source": pk["source"] + " (burst copy)",
                                     "traffic": None, "kernel_ms": round(r0["us"] / 1e3, 5)},
                        "gpu_launches": r0["timed_launches"], "clocks": clk.summary(), "more": kq[1:]})
        else:
            out["kquants"] = {"rows": kq, "clocks": clk.summary()}

    if args.workload in ("headline", "peaks"):
        barrier()
        pr = peak_probes(torch, stream, local_rank, sms)
        if args.workload == "peaks":
            k2 = pr["tcgen05.mma kind::f16 128x256x16"]
            out.update({"value": k2["tera_ops_per_s"], "unit": "TFLOP/s", "ms_per_step": k2["ms"], "dtype": "f16",
                        "config": {"workload": "throughput probes"}, "clocks": pr["clocks"], "peaks": pr,
                        "gpu_launches": 22})
        else:
            out["peaks"] = pr
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))
    return 0


def e2e(torch, wl, steps, warmup):
    """Same metric through the public API with host buffers: each step copies
    the step's activations from pinned host memory (one copy: the inputs share
    one device buffer), runs every call of the path and reads every output back
    to pinned host memory (one copy).  Measured two ways: the
    step replayed from a CUDA graph holding the copies and the calls (how an
    engine runs a decode step; the copies still move every byte every step),
    and eagerly from Python (no graph).  The graph figure is the line's value."""
    # every input of the step in one device buffer and every output in
    # another (the calls get views of them, as an engine that owns its
    # activation buffers would), so a step moves them with one copy each way
    def gather(tensors):
        flat = torch.empty(sum(t.numel() for t in tensors), dtype=torch.float32, device="cuda")
        views, o = [], 0
        for t in tensors:
            v = flat[o:o + t.numel()].view_as(t)
            v.copy_(t)
            views.append(v)
            o += t.numel()
        return flat, views

    keys = list(wl.x)
    dx, xv = gather([wl.x[k] for k in keys])
    for k, v in zip(keys, xv):
        wl.x[k] = v
    outs = [(p, j) for p in wl.y for j in (0, 1) if wl.y[p][j] is not None]
    dy, yv = gather([wl.y[p][j] for p, j in outs])
    ynew = {p: [None, None] for p in wl.y}
    for (p, j), v in zip(outs, yv):
        ynew[p][j] = v
    wl.y = {p: tuple(v) for p, v in ynew.items()}
    hx = dx.cpu().pin_memory()
    hy = torch.empty(dy.numel(), dtype=torch.float32).pin_memory()

    # the copies run on the SMs (zq_copy: one short round trip per thread
    # over the host link instead of a copy engine's start-up); the copy
    # engines' figure (cudaMemcpyAsync through torch) is kept beside it
    def step(r, s, sm_copy=True):
        if sm_copy:
            wl.zq.copy(dx, hx, stream=s)
        else:
            dx.copy_(hx, non_blocking=True)
        wl.run(r, stream=s)
        if sm_copy:
            wl.zq.copy(hy, dy, stream=s)
        else:
            hy.copy_(dy, non_blocking=True)

    def timed(run_one):
        for i in range(warmup):
            run_one(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(steps):
            run_one(i)
        e1.record()
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) / steps
        return max(e0.elapsed_time(e1) / steps, wall * 1e3)

    s = torch.cuda.current_stream()
    ms_eager = timed(lambda i: step(i % wl.R, s))
    side = torch.cuda.Stream()

    def graphs_of(sm_copy):
        out = []
        for r in range(wl.R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                step(r, torch.cuda.current_stream(), sm_copy)
            out.append(g)
        return out

    graphs = graphs_of(True)
    ms_graph = timed(lambda i: graphs[i % wl.R].replay())
    graphs_dma = graphs_of(False)
    ms_dma = timed(lambda i: graphs_dma[i % wl.R].replay())
    gbs = lambda ms: round(wl.algo_bytes() / (ms * 1e-3) / 1e9, 1)
    return {"value": gbs(ms_graph), "unit": "GB/s", "ms_per_step": round(ms_graph, 5),
            "h2d_bytes_per_step": int(wl.input_bytes()), "d2h_bytes_per_step": int(wl.output_bytes()),
            "graph": True, "copies": "zq_copy (SM copy kernels, pinned host buffers)",
            "eager": {"value": gbs(ms_eager), "ms_per_step": round(ms_eager, 5)},
            "copy_engines": {"value": gbs(ms_dma), "ms_per_step": round(ms_dma, 5)}}


def run_reference(args):
    """The oracle as it stands, on the host cores (single thread)."""
    shapes = inputs.LAYER_27B
    per_step = []
    # each step: a bounded sample of the decode layer, scaled to a full step
    for i in range(args.warmup + args.steps):
        secs, sample = oracle_sample(shapes, 1, budget_s=1.0, seed=0)
        if i >= args.warmup:
            per_step.append(secs)
    secs = statistics.mean(per_step) if per_step else float("nan")
    v = layer_algo_bytes(shapes, 1) / secs / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic", "config": decode_config("decode-27b-layer", shapes),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"per step: {sample}, scaled to a full step"},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
