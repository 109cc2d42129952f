"""Benchmark of the differential-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-rows] [--no-cpu-baseline]

Prints ONE JSON line (rank 0).  `value` is the throughput of the selected
workload (default: V1 forward bf16, B4 H12 N4096 d_qk 128 d_v 256, causal)
with inputs resident in HBM; `rows` holds the same measurement for every
other step of the path (V1 fp32, V2 gate + forward, V2 decode, V1
forward + backward, deterministic V1 backward, V2 forward + backward, V1
decode, grouped attention) on its own workload; `e2e` repeats the main
workload through the public API with every step's inputs uploaded from pinned
host memory and its results read back inside the timed region (uploads,
kernels and read-backs of consecutive steps overlap on three streams; decode
keeps its KV cache resident as model state); `roofline` relates the dominant kernel's live CUDA-event time
to the measured (or fallback) peak; `cpu_baseline` times the fp64 oracle on a
bounded sample of the same workload.

`--impl reference` times the fp64 CPU oracle (the only reference there is)
as the reference arm on the same workload and metric.

Multi-GPU (torchrun): replicas only — every rank runs the full workload on
its own GPU (no collective on the data path); the timed region is bracketed
by barriers and the slowest rank's time is reported (weak scaling).
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# --------------------------------------------------------------- workloads --
# Algorithmic work per call (causal: half of the N^2 score matrix, the
# flash-attention convention).


def v1_fwd_flops(B, N, H, dqk, dv):
    return B * H * 0.5 * (4.0 * N * N * dqk + 2.0 * N * N * dv)


def v1_bwd_flops(B, N, H, dqk, dv):
    return B * H * 0.5 * (12.0 * N * N * dqk + 4.0 * N * N * dv)


def v2_fwd_flops(B, N, h, d):
    return B * 2 * h * 0.5 * 4.0 * N * N * d


def v2_bwd_flops(B, N, h, d):
    return B * 2 * h * 0.5 * 10.0 * N * N * d


def decode_bytes(B, L, hkv, d):
    return 2.0 * B * L * hkv * d * 2


def v1_decode_bytes(B, L, H, dqk, dv):
    return B * L * H * (2.0 * dqk + dv) * 2


class Workload:
    """One step of the path on its configuration."""

    name = ""
    desc = ""
    unit = "TFLOP/s"
    bound = "tensor"
    dtype = "bf16"
    launches = 1

    def work(self):  # flops or bytes per step
        raise NotImplementedError

    def setup(self, dev):
        raise NotImplementedError

    def run(self):  # device-resident step
        raise NotImplementedError

    def run_dominant(self):  # the dominant kernel alone (for the roofline)
        self.run()

    def dominant_work(self):
        return self.work()

    def scale(self, seconds):
        w = self.work()
        return w / seconds / (1e12 if self.unit == "TFLOP/s" else 1e9)


class V1Fwd(Workload):
    name = "v1_fwd"
    desc = "V1 DiffAttn fwd bf16 B4 H12 N4096 d_qk128 d_v256 causal, layer 1"
    B, N, H, dqk, dv, layer = 4, 4096, 12, 128, 256, 1

    def work(self):
        return v1_fwd_flops(self.B, self.N, self.H, self.dqk, self.dv)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.v1_inputs(self.B, self.N, self.H, self.dqk, self.dv, "bf16", seed=1002,
                                 device=dev)
        self.li = bd.diffattn_lambda_init(self.layer)
        self.out = torch.empty((self.B, self.N, self.H, self.dv), dtype=torch.bfloat16, device=dev)
        need = bd.load().diffattn_v1_fwd_workspace_size(self.B, self.N, self.H, self.dqk, self.dv, 1)
        self.fws = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)

    def args(self, t):
        return [t[n] for n in ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")]

    def setup_host(self):
        """Inputs for the oracle legs alone: drawn on the host with the same
        shapes and distributions (the host generator's values differ from the
        device's; the oracle's time does not depend on them), lambda_init from
        the oracle; nothing of the library is loaded."""
        from differential_attention_diff_gb300 import synth
        from oracle import diffattn_oracle as orc
        self.t = synth.v1_inputs(self.B, self.N, self.H, self.dqk, self.dv,
                                 "f32" if self.dtype == "f32" else "bf16", seed=1002, device="cpu",
                                 with_dy=True)
        self.li = float(np.float32(orc.lambda_init(self.layer)))

    def run(self):
        self.bd.diffattn_v1_fwd(*self.args(self.t), self.li, out=self.out, workspace=self.fws)

    # end-to-end through the public API with host buffers
    # end-to-end through the public API: inputs uploaded from pinned host
    # memory, the result read back, every step (see run_e2e)
    def e2e_inputs(self):
        return dict(self.t)

    def e2e_outputs(self):
        return [self.out]

    def e2e_compute(self, d, outs):
        self.bd.diffattn_v1_fwd(*self.args(d), self.li, out=outs[0], workspace=self.fws)

    def oracle_sample(self, big=True):
        """fp64 oracle on a bounded sample (every head of the first batches, a
        seeded set of query rows); returns (seconds, flops of the sampled
        rows, description)."""
        from oracle import diffattn_oracle as orc
        nb, nrows = (min(self.B, 4), min(self.N, 1024)) if big else (1, min(self.N, 128))
        rows = np.sort(np.random.default_rng(0).choice(self.N, nrows, replace=False))
        ts = {k: v[:nb].to("cpu", torch.float64).numpy() if v.dim() == 4 else
              v.to("cpu", torch.float64).numpy() for k, v in self.t.items()}
        t0 = time.perf_counter()
        orc.v1_forward(*(ts[n] for n in ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")),
                       self.li, rows=rows)
        dt = time.perf_counter() - t0
        keys = float(np.sum(rows + 1))  # causal keys of the sampled rows
        flops = nb * self.H * keys * (4.0 * self.dqk + 2.0 * self.dv)
        return dt, flops, (f"batches 0-{nb - 1}, {self.H} heads, {nrows} seeded query rows of "
                           f"{self.N} (fp64 numpy oracle)")


class V1FwdBwd(V1Fwd):
    name = "v1_fwd_bwd"
    desc = "V1 DiffAttn fwd+bwd bf16 B1 H16 N8192 d_qk128 d_v256 causal, layer 1"
    B, N, H, dqk, dv, layer = 1, 8192, 16, 128, 256, 1
    deterministic = False

    def work(self):
        return v1_fwd_flops(self.B, self.N, self.H, self.dqk, self.dv) + \
            v1_bwd_flops(self.B, self.N, self.H, self.dqk, self.dv)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.v1_inputs(self.B, self.N, self.H, self.dqk, self.dv, "bf16", seed=1005,
                                 device=dev, with_dy=True)
        self.li = bd.diffattn_lambda_init(self.layer)
        self.out = torch.empty((self.B, self.N, self.H, self.dv), dtype=torch.bfloat16, device=dev)
        need = bd.load().diffattn_v1_fwd_workspace_size(self.B, self.N, self.H, self.dqk, self.dv, 1)
        self.fws = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
        _, self.saves = bd.diffattn_v1_fwd(*self.args(self.t), self.li, out=self.out, save=True,
                                           workspace=self.fws)
        self.grads = bd.diffattn_v1_bwd(*self.args(self.t), self.li, self.out, self.t["dy"],
                                        self.saves, deterministic=self.deterministic)
        need = bd.load().diffattn_v1_bwd_workspace_size(self.B, self.N, self.H, self.dqk, self.dv,
                                                        int(self.deterministic))
        self.ws = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
        self.launches = None

    def run(self):
        self.bd.diffattn_v1_fwd(*self.args(self.t), self.li, out=self.out, save=True,
                                saves=self.saves, workspace=self.fws)
        self.bd.diffattn_v1_bwd(*self.args(self.t), self.li, self.out, self.t["dy"], self.saves,
                                grads=self.grads, workspace=self.ws,
                                deterministic=self.deterministic)

    def run_dominant(self):
        self.bd.diffattn_v1_bwd(*self.args(self.t), self.li, self.out, self.t["dy"], self.saves,
                                grads=self.grads, workspace=self.ws,
                                deterministic=self.deterministic)

    def dominant_work(self):
        return v1_bwd_flops(self.B, self.N, self.H, self.dqk, self.dv)


    GRADS = ("dq1", "dq2", "dk1", "dk2", "dv", "dlq1", "dlk1", "dlq2", "dlk2")

    def e2e_inputs(self):
        return dict(self.t)

    def e2e_outputs(self):
        return [self.grads[n] for n in self.GRADS]

    def e2e_compute(self, d, outs):
        self.bd.diffattn_v1_fwd(*self.args(d), self.li, out=self.out, save=True, saves=self.saves,
                                workspace=self.fws)
        self.bd.diffattn_v1_bwd(*self.args(d), self.li, self.out, d["dy"], self.saves,
                                grads=dict(zip(self.GRADS, outs)), workspace=self.ws,
                                deterministic=self.deterministic)


    def oracle_sample(self, big=True):
        """fp64 oracle forward + backward on a bounded sample: one head of the
        workload cut to its first n tokens (causal, so a prefix is a
        self-contained problem)."""
        from oracle import diffattn_oracle as orc
        n = 2048 if big else 512
        names = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
        ts = {k: (v[0:1, :n, 0:1] if v.dim() == 4 else v).to("cpu", torch.float64).numpy()
              for k, v in self.t.items()}
        t0 = time.perf_counter()
        orc.v1_forward(*(ts[k] for k in names), self.li)
        orc.v1_backward(*(ts[k] for k in names), self.li, ts["dy"])
        dt = time.perf_counter() - t0
        flops = v1_fwd_flops(1, n, 1, self.dqk, self.dv) + v1_bwd_flops(1, n, 1, self.dqk, self.dv)
        return dt, flops, f"batch 0, head 0, first {n} tokens (fp64 oracle fwd+bwd)"


class V1FwdBwdDet(V1FwdBwd):
    name = "v1_fwd_bwd_det"
    desc = ("V1 DiffAttn fwd+bwd bf16 B1 H16 N8192 d_qk128 d_v256 causal, layer 1, "
            "deterministic dQ (bitwise reproducible)")
    deterministic = True


class V1FwdF32(V1Fwd):
    name = "v1_fwd_f32"
    desc = "V1 DiffAttn fwd fp32 B1 H2 N64 d_qk16 d_v32 causal, layer 1 (latency-bound)"
    dtype = "f32"
    bound = "alu"
    B, N, H, dqk, dv, layer = 1, 64, 2, 16, 32, 1

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.v1_inputs(self.B, self.N, self.H, self.dqk, self.dv, "f32", seed=1001,
                                 device=dev)
        self.li = bd.diffattn_lambda_init(self.layer)
        self.out = torch.empty((self.B, self.N, self.H, self.dv), dtype=torch.float32, device=dev)
        self.fws = None


class V2Fwd(Workload):
    name = "v2_fwd"
    desc = "V2 DiffAttn fwd bf16 B2 N8192 64q/8kv heads d128 causal, gate from X[2,8192,4096]"
    launches = 2
    B, N, h, hkv, d, dm = 2, 8192, 32, 8, 128, 4096

    def work(self):
        return v2_fwd_flops(self.B, self.N, self.h, self.d)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.v2_inputs(self.B, self.N, self.h, self.hkv, self.d, self.dm, seed=1003,
                                 device=dev)
        self.out = torch.empty((self.B, self.N, self.h, self.d), dtype=torch.bfloat16, device=dev)
        need = bd.load().diffattn_v2_fwd_workspace_size(self.B, self.N, self.h, 0)
        self.ws = torch.empty((need,), dtype=torch.uint8, device=dev)
        self.gate = bd.diffattn_v2_gate(self.t["x"], self.t["w_lambda"])

    def run(self):
        t = self.t
        self.bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"],
                                out=self.out, workspace=self.ws)

    def setup_host(self):
        """Inputs for the oracle legs alone, drawn on the host (see V1Fwd)."""
        from differential_attention_diff_gb300 import synth
        self.t = synth.v2_inputs(self.B, self.N, self.h, self.hkv, self.d, self.dm, seed=1003,
                                 device="cpu", with_dout=True)

    def run_dominant(self):
        t = self.t
        self.bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], gate=self.gate, out=self.out)

    def e2e_inputs(self):
        return dict(self.t)

    def e2e_outputs(self):
        return [self.out]

    def e2e_compute(self, d, outs):
        self.bd.diffattn_v2_fwd(d["q"], d["k"], d["v"], x=d["x"], w_lambda=d["w_lambda"],
                                out=outs[0], workspace=self.ws)

    def oracle_sample(self, big=True):
        from oracle import diffattn_oracle as orc
        rows = np.sort(np.random.default_rng(0).choice(self.N, 256 if big else 48, replace=False))
        G = 2 * self.h // self.hkv
        t0 = time.perf_counter()
        for p in range(4):  # four pairs of batch 0 (one per K/V group of the first four)
            g = (2 * p) // G
            sl = lambda x, a, b: x[0:1, :, a:b].to("cpu", torch.float64).numpy()  # noqa: E731
            gate = orc.v2_gate(self.t["x"][0:1].to("cpu", torch.float64).numpy(),
                               self.t["w_lambda"][:, p:p + 1].to("cpu", torch.float64).numpy())
            orc.v2_forward(sl(self.t["q"], 2 * p, 2 * p + 2), sl(self.t["k"], g, g + 1),
                           sl(self.t["v"], g, g + 1), gate, rows=rows)
        dt = time.perf_counter() - t0
        flops = 4 * 2 * float(np.sum(rows + 1)) * 4.0 * self.d
        return dt, flops, f"batch 0, 4 pairs, {len(rows)} seeded query rows of 8192 (gate included)"


class V2FwdBwd(V2Fwd):
    name = "v2_fwd_bwd"
    desc = ("V2 DiffAttn fwd+bwd bf16 B2 N8192 64q/8kv heads d128 causal, gate from X[2,8192,4096]; "
            "grads of q, k, v, X, W_lambda")
    launches = None

    def work(self):
        return v2_fwd_flops(self.B, self.N, self.h, self.d) + v2_bwd_flops(self.B, self.N, self.h, self.d)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.v2_inputs(self.B, self.N, self.h, self.hkv, self.d, self.dm, seed=1003,
                                 device=dev, with_dout=True)
        self.out = torch.empty((self.B, self.N, self.h, self.d), dtype=torch.bfloat16, device=dev)
        need = bd.load().diffattn_v2_fwd_workspace_size(self.B, self.N, self.h, 0)
        self.ws = torch.empty((need,), dtype=torch.uint8, device=dev)
        t = self.t
        _, self.saves = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"],
                                           out=self.out, save=True, workspace=self.ws)
        need = bd.diffattn_v2_bwd_workspace_size(self.B, self.N, self.h, self.dm)
        self.bws = torch.empty((need,), dtype=torch.uint8, device=dev)
        self.grads = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], self.saves, x=t["x"],
                                        w_lambda=t["w_lambda"], workspace=self.bws)

    def _step(self, t):
        self.bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], out=self.out,
                                save=True, saves=self.saves, workspace=self.ws)
        self.bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], self.saves, x=t["x"],
                                w_lambda=t["w_lambda"], grads=self.grads, workspace=self.bws)

    def run(self):
        self._step(self.t)

    def run_dominant(self):
        t = self.t
        self.bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], self.saves, x=t["x"],
                                w_lambda=t["w_lambda"], grads=self.grads, workspace=self.bws)

    def dominant_work(self):
        return v2_bwd_flops(self.B, self.N, self.h, self.d)

    def e2e_inputs(self):
        return dict(self.t)

    def e2e_outputs(self):
        return [self.grads[n] for n in sorted(self.grads)]

    def e2e_compute(self, d, outs):
        t = d
        self.bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], out=self.out,
                                save=True, saves=self.saves, workspace=self.ws)
        self.bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], self.saves, x=t["x"],
                                w_lambda=t["w_lambda"], grads=dict(zip(sorted(self.grads), outs)),
                                workspace=self.bws)

    def oracle_sample(self, big=True):
        """fp64 oracle backward on a bounded sample: one (batch, K/V group) of
        the workload cut to its first n tokens (causal, so a prefix is a
        self-contained problem)."""
        from oracle import diffattn_oracle as orc
        n = 1024 if big else 256
        G = 2 * self.h // self.hkv
        sl = lambda x: x.to("cpu", torch.float64).numpy()  # noqa: E731
        t = self.t
        t0 = time.perf_counter()
        orc.v2_backward(sl(t["q"][0:1, :n, 0:G]), sl(t["k"][0:1, :n, 0:1]), sl(t["v"][0:1, :n, 0:1]),
                        sl(t["x"][0:1, :n]), sl(t["w_lambda"][:, 0:G // 2]), sl(t["dout"][0:1, :n, 0:G // 2]))
        dt = time.perf_counter() - t0
        flops = v2_fwd_flops(1, n, G // 2, self.d) + v2_bwd_flops(1, n, G // 2, self.d)
        return dt, flops, f"batch 0, K/V group 0 ({G} query heads), first {n} tokens (fp64 oracle fwd+bwd)"


class GroupedFwd(Workload):
    name = "grouped_fwd"
    desc = ("Grouped DiffAttn 3:1 fwd bf16 B2 N8192, 64 query heads = 16 x (3 signal + 1 noise), 8 kv heads, "
            "d128 causal, gate from X[2,8192,4096]")
    launches = 3
    B, N, h, ratio, hkv, d, dm = 2, 8192, 48, 3, 8, 128, 4096

    def work(self):
        Hq = self.h // self.ratio * (self.ratio + 1)
        return v2_fwd_flops(self.B, self.N, Hq // 2, self.d)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.grouped_inputs(self.B, self.N, self.h, self.ratio, self.hkv, self.d, self.dm, seed=1007,
                                      device=dev)
        self.out = torch.empty((self.B, self.N, self.h, self.d), dtype=torch.bfloat16, device=dev)
        need = bd.load().diffattn_grouped_fwd_workspace_size(self.B, self.N, self.h, self.ratio, self.d, 0, 0)
        self.ws = torch.empty((need,), dtype=torch.uint8, device=dev)

    def run(self):
        t = self.t
        self.bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], self.ratio, x=t["x"], w_lambda=t["w_lambda"],
                                     out=self.out, workspace=self.ws)

    def setup_host(self):
        """Inputs for the oracle legs alone, drawn on the host (see V1Fwd)."""
        from differential_attention_diff_gb300 import synth
        self.t = synth.grouped_inputs(self.B, self.N, self.h, self.ratio, self.hkv, self.d, self.dm, seed=1007,
                                      device="cpu")

    def e2e_inputs(self):
        return dict(self.t)

    def e2e_outputs(self):
        return [self.out]

    def e2e_compute(self, d, outs):
        self.bd.diffattn_grouped_fwd(d["q"], d["k"], d["v"], self.ratio, x=d["x"], w_lambda=d["w_lambda"],
                                     out=outs[0], workspace=self.ws)

    def oracle_sample(self, big=True):
        from oracle import diffattn_oracle as orc
        rows = np.sort(np.random.default_rng(0).choice(self.N, 256 if big else 48, replace=False))
        sl = lambda x: x.to("cpu", torch.float64).numpy()  # noqa: E731
        t = self.t
        t0 = time.perf_counter()
        gate = orc.v2_gate(sl(t["x"][0:1]), sl(t["w_lambda"][:, 0:self.ratio]))
        orc.grouped_forward(sl(t["q"][0:1, :, 0:self.ratio + 1]), sl(t["k"][0:1, :, 0:1]), sl(t["v"][0:1, :, 0:1]),
                            gate, self.ratio, rows=rows)
        dt = time.perf_counter() - t0
        flops = (self.ratio + 1) * float(np.sum(rows + 1)) * 4.0 * self.d
        return dt, flops, f"batch 0, group 0 ({self.ratio + 1} query heads), {len(rows)} seeded rows (gate included)"


class GroupedFwdBwd(GroupedFwd):
    name = "grouped_fwd_bwd"
    desc = ("Grouped DiffAttn 3:1 fwd+bwd bf16 B2 N8192, 64 query heads = 16 x (3 signal + 1 noise), 8 kv heads, "
            "d128 causal, gate from X[2,8192,4096]; grads of q, k, v, X, W_lambda")
    launches = None

    def work(self):
        Hq = self.h // self.ratio * (self.ratio + 1)
        return v2_fwd_flops(self.B, self.N, Hq // 2, self.d) + v2_bwd_flops(self.B, self.N, Hq // 2, self.d)

    def dominant_work(self):
        Hq = self.h // self.ratio * (self.ratio + 1)
        return v2_bwd_flops(self.B, self.N, Hq // 2, self.d)

    def setup(self, dev):
        super().setup(dev)
        t = self.t
        g = torch.Generator(device=dev).manual_seed(1008)
        t["dout"] = torch.randn((self.B, self.N, self.h, self.d), generator=g, device=dev).to(torch.bfloat16)
        Hq = self.h // self.ratio * (self.ratio + 1)
        self.saves = dict(o_heads=torch.empty((self.B, self.N, Hq, self.d), dtype=torch.bfloat16, device=dev),
                          lse=torch.empty((self.B, Hq, self.N), dtype=torch.float32, device=dev))
        need = self.bd.load().diffattn_grouped_fwd_workspace_size(self.B, self.N, self.h, self.ratio, self.d, 0, 1)
        self.ws = torch.empty((need,), dtype=torch.uint8, device=dev)
        self._fwd(t)
        need = self.bd.diffattn_grouped_bwd_workspace_size(self.B, self.N, self.h, self.ratio, self.dm)
        self.bws = torch.empty((need,), dtype=torch.uint8, device=dev)
        self.grads = self.bd.diffattn_grouped_bwd(t["q"], t["k"], t["v"], t["dout"], self.saves, self.ratio,
                                                  x=t["x"], w_lambda=t["w_lambda"], workspace=self.bws)

    def _fwd(self, t):
        self.bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], self.ratio, x=t["x"], w_lambda=t["w_lambda"],
                                     out=self.out, o_heads=self.saves["o_heads"], lse=self.saves["lse"],
                                     workspace=self.ws)

    def _bwd(self, t, grads):
        self.bd.diffattn_grouped_bwd(t["q"], t["k"], t["v"], t["dout"], self.saves, self.ratio, x=t["x"],
                                     w_lambda=t["w_lambda"], grads=grads, workspace=self.bws)

    def run(self):
        self._fwd(self.t)
        self._bwd(self.t, self.grads)

    def run_dominant(self):
        self._bwd(self.t, self.grads)

    def e2e_outputs(self):
        return [self.grads[n] for n in sorted(self.grads)]

    def e2e_compute(self, d, outs):
        self._fwd(d)
        self._bwd(d, dict(zip(sorted(self.grads), outs)))

    def setup_host(self):
        super().setup_host()
        g = torch.Generator().manual_seed(1008)
        self.t["dout"] = torch.randn((self.B, self.N, self.h, self.d), generator=g).to(torch.bfloat16)

    def oracle_sample(self, big=True):
        """fp64 oracle forward + backward on a bounded sample: one (batch, K/V
        group) of the workload cut to its first n tokens (causal, so a prefix
        is a self-contained problem)."""
        from oracle import diffattn_oracle as orc
        n = 1024 if big else 256
        Hq = self.h // self.ratio * (self.ratio + 1)
        G = Hq // self.hkv
        hg = G // (self.ratio + 1) * self.ratio  # output heads of the group
        sl = lambda x: x.to("cpu", torch.float64).numpy()  # noqa: E731
        t = self.t
        t0 = time.perf_counter()
        orc.grouped_backward(sl(t["q"][0:1, :n, 0:G]), sl(t["k"][0:1, :n, 0:1]), sl(t["v"][0:1, :n, 0:1]),
                             sl(t["x"][0:1, :n]), sl(t["w_lambda"][:, 0:hg]), sl(t["dout"][0:1, :n, 0:hg]),
                             self.ratio)
        dt = time.perf_counter() - t0
        flops = v2_fwd_flops(1, n, G // 2, self.d) + v2_bwd_flops(1, n, G // 2, self.d)
        return dt, flops, f"batch 0, K/V group 0 ({G} query heads), first {n} tokens (fp64 oracle fwd+bwd)"


class V2Decode(Workload):
    name = "v2_decode"
    desc = "V2 decode bf16 B64 cache 32768 8 KV heads 64 query heads d128, gate from X[64,4096]"
    unit = "GB/s"
    bound = "hbm"
    launches = 3
    B, L, h, hkv, d, dm = 64, 32768, 32, 8, 128, 4096

    def work(self):
        return decode_bytes(self.B, self.L, self.hkv, self.d)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.decode_inputs(self.B, self.L, self.h, self.hkv, self.d, self.dm, seed=1004,
                                     device=dev)
        self.out = torch.empty((self.B, self.h, self.d), dtype=torch.bfloat16, device=dev)
        need = bd.diffattn_v2_decode_workspace_size(self.B, self.h, self.hkv, self.d, self.L)
        self.ws = torch.empty((need,), dtype=torch.uint8, device=dev)

    def run(self):
        t = self.t
        self.bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], x=t["x"],
                                   w_lambda=t["w_lambda"], out=self.out, workspace=self.ws)

    def setup_host(self):
        """Inputs for the oracle legs alone, drawn on the host (see V1Fwd):
        only the sequence the oracle sample reads (a full 32768-position
        cache), not all 64."""
        from differential_attention_diff_gb300 import synth
        self.t = synth.decode_inputs(1, self.L, self.h, self.hkv, self.d, self.dm, seed=1004, device="cpu")

    # end to end: the KV cache is the model's resident state; each step
    # uploads the new tokens' queries and gate inputs and reads the output
    RESIDENT = ("k_cache", "v_cache", "seqlens")

    def e2e_inputs(self):
        return {k: v for k, v in self.t.items() if k not in self.RESIDENT}

    def e2e_outputs(self):
        return [self.out]

    def e2e_compute(self, d, outs):
        t = self.t
        self.bd.diffattn_v2_decode(d["q"], t["k_cache"], t["v_cache"], x=d["x"], w_lambda=d["w_lambda"],
                                   out=outs[0], workspace=self.ws)

    def oracle_sample(self, big=True):
        from oracle import diffattn_oracle as orc
        t0 = time.perf_counter()
        b = 0
        gate = orc.v2_gate(self.t["x"][b:b + 1].to("cpu", torch.float64).numpy(),
                           self.t["w_lambda"].to("cpu", torch.float64).numpy())
        orc.v2_decode(self.t["q"][b:b + 1].to("cpu", torch.float64).numpy(),
                      self.t["k_cache"][b:b + 1].to("cpu", torch.float64).numpy(),
                      self.t["v_cache"][b:b + 1].to("cpu", torch.float64).numpy(), [self.L], gate)
        dt = time.perf_counter() - t0
        return dt, decode_bytes(1, self.L, self.hkv, self.d), "sequence 0 of 64 (full cache)"


class V1Decode(Workload):
    name = "v1_decode"
    desc = "V1 decode bf16 B64 cache 32768 16 heads d_qk128 d_v256 (K1, K2 and V caches), layer 1"
    unit = "GB/s"
    bound = "hbm"
    launches = 2
    B, L, H, dqk, dv, layer = 64, 32768, 16, 128, 256, 1

    def work(self):
        return v1_decode_bytes(self.B, self.L, self.H, self.dqk, self.dv)

    def setup(self, dev):
        from differential_attention_diff_gb300 import binding as bd, synth
        self.bd = bd
        self.t = synth.v1_decode_inputs(self.B, self.L, self.H, self.dqk, self.dv, seed=1006, device=dev)
        self.li = bd.diffattn_lambda_init(self.layer)
        self.out = torch.empty((self.B, self.H, self.dv), dtype=torch.bfloat16, device=dev)
        need = bd.diffattn_v1_decode_workspace_size(self.B, self.H, self.dv, self.L)
        self.ws = torch.empty((need,), dtype=torch.uint8, device=dev)

    def run(self):
        t = self.t
        self.bd.diffattn_v1_decode(t["q1"], t["q2"], t["k1_cache"], t["k2_cache"], t["v_cache"],
                                   t["lq1"], t["lk1"], t["lq2"], t["lk2"], self.li, out=self.out,
                                   workspace=self.ws)

    def setup_host(self):
        """Inputs for the oracle legs alone, drawn on the host (see V1Fwd):
        only the sequence the oracle sample reads."""
        from differential_attention_diff_gb300 import synth
        from oracle import diffattn_oracle as orc
        self.t = synth.v1_decode_inputs(1, self.L, self.H, self.dqk, self.dv, seed=1006, device="cpu")
        self.li = float(np.float32(orc.lambda_init(self.layer)))

    RESIDENT = ("k1_cache", "k2_cache", "v_cache", "seqlens")

    def e2e_inputs(self):
        return {k: v for k, v in self.t.items() if k not in self.RESIDENT}

    def e2e_outputs(self):
        return [self.out]

    def e2e_compute(self, d, outs):
        t = self.t
        self.bd.diffattn_v1_decode(d["q1"], d["q2"], t["k1_cache"], t["k2_cache"], t["v_cache"], d["lq1"],
                                   d["lk1"], d["lq2"], d["lk2"], self.li, out=outs[0], workspace=self.ws)

    def oracle_sample(self, big=True):
        from oracle import diffattn_oracle as orc
        t = self.t
        sl = lambda x: x[0:1].to("cpu", torch.float64).numpy()  # noqa: E731
        lam = [t[n].to("cpu", torch.float64).numpy() for n in ("lq1", "lk1", "lq2", "lk2")]
        t0 = time.perf_counter()
        orc.v1_decode(sl(t["q1"]), sl(t["q2"]), sl(t["k1_cache"]), sl(t["k2_cache"]), sl(t["v_cache"]),
                      [self.L], *lam, self.li)
        dt = time.perf_counter() - t0
        return dt, v1_decode_bytes(1, self.L, self.H, self.dqk, self.dv), "sequence 0 of 64 (full cache)"


class V2DecodeSmall(V2Decode):
    """The decode kernel on a 1 GB cache (B8): big enough that DRAM figures
    mean something, small enough for a multi-pass ncu capture."""
    name = "v2_decode_small"
    desc = "V2 decode bf16 B8 cache 32768 8 KV heads 64 query heads d128 (profiling size)"
    B = 8


class V2FwdBwdSmall(V2FwdBwd):
    """The V2 training step at B1 N4096 (134 MB of dQ accumulators, above L2):
    a size for multi-pass ncu captures of the backward's kernels."""
    name = "v2_fwd_bwd_small"
    desc = "V2 DiffAttn fwd+bwd bf16 B1 N4096 64q/8kv heads d128 causal (profiling size)"
    B, N = 1, 4096


class V1DecodeSmall(V1Decode):
    """The V1 decode kernels on a 2.1 GB cache (B4): above L2, small enough
    for a multi-pass ncu capture."""
    name = "v1_decode_small"
    desc = "V1 decode bf16 B4 cache 32768 16 heads d_qk128 d_v256 (profiling size)"
    B = 4


WORKLOADS = {w.name: w for w in (V1Fwd, V1FwdF32, V2Fwd, V2Decode, V1FwdBwd, V1FwdBwdDet, V2FwdBwd,
                                 V1Decode, GroupedFwd, GroupedFwdBwd)}
PROFILE_ONLY = {V2DecodeSmall.name: V2DecodeSmall, V2FwdBwdSmall.name: V2FwdBwdSmall,
                V1DecodeSmall.name: V1DecodeSmall}

# ----------------------------------------------------------------- helpers --


KERNEL_SOURCES = {
    "v1_fwd": ("v1_fwd.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
    "v1_fwd_bwd": ("v1_bwd.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
    "v1_fwd_bwd_det": ("v1_bwd.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
    "v2_fwd": ("v2_fwd.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
    "v2_decode": ("decode.cu", "common.cuh"),
    "v2_fwd_bwd": ("v2_bwd.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
    "v1_decode": ("v1_decode.cu", "common.cuh"),
    "grouped_fwd": ("v2_fwd.cu", "grouped.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
    "grouped_fwd_bwd": ("v2_bwd.cu", "softmax.cuh", "tma.cuh", "common.cuh"),
}


def source_hash(workload):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(workload, ()):
        with open(os.path.join(ROOT, "differential_attention_diff_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    record (profiles/traffic.json), or None when the kernel's sources changed
    since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(path)).get(workload)
    except Exception:  # noqa: BLE001
        return None
    if not rec or rec.get("source_hash") != source_hash(workload):
        return None
    return rec.get("dram_bytes_per_launch")


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            return d, "measured"
        except Exception:  # noqa: BLE001
            pass
    return {}, "fallback"


def peak_for(bound, long_step=False):
    d, src = measured_peaks()
    if bound == "hbm":
        v = d.get("hbm_gbs")
        return (float(v), "of measured") if v else (FALLBACK_HBM_GBS, "of fallback")
    if bound == "tensor":
        key = "bf16_tflops_sustained" if long_step else "bf16_tflops"
        v = d.get(key) or d.get("bf16_tflops")
        return (float(v), "of measured") if v else (FALLBACK_BF16_TFLOPS, "of fallback")
    return None, None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        """Start sampling every 50 ms and return once the first sample is in
        (at most 3 s), so that a short timed region is bracketed by samples."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:  # noqa: BLE001
            self.proc = None
            return
        t0 = time.time()
        while not self.lines and self.proc.poll() is None and time.time() - t0 < 3.0:
            time.sleep(0.005)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        # one more sample after the region ends (at most 1 s): the timed
        # region can be shorter than the sampling interval
        n0, t0 = len(self.lines), time.time()
        while len(self.lines) <= n0 and self.proc.poll() is None and time.time() - t0 < 1.0:
            time.sleep(0.005)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "every 50 ms from just before the timed region to just after it"}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(total_ms, steps, work_per_step, unit_scale, ws, device):
    """Whole-job throughput of `ws` replicas: the slowest rank's time (max
    over ranks of the local timed total), the work of every rank summed.
    Returns (ms_per_step, value)."""
    if ws > 1:
        import torch.distributed as dist
        t = torch.tensor([total_ms], device=device, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms = total_ms / steps
    return ms, work_per_step * ws / (ms / 1e3) / unit_scale


def run_e2e(main, steps, warm=2, n_up=1):
    """End-to-end steps through the public API.  Every step uploads its
    inputs from pinned host memory, runs the call and reads its outputs back
    into pinned host memory.  Two device buffer sets and three streams
    (upload, compute, download) let step i+1's upload and step i-1's download
    run under step i's kernels, as a serving loop would; every step still
    moves all of its bytes inside the timed region.  Returns (ms per step,
    h2d bytes per step, d2h bytes per step)."""
    src = main.e2e_inputs()
    tmpl = main.e2e_outputs()
    host_in = {k: v.cpu().pin_memory() for k, v in src.items()}
    dev_in = [{k: torch.empty_like(v) for k, v in src.items()} for _ in range(2)]
    dev_out = [[torch.empty_like(t) for t in tmpl] for _ in range(2)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in tmpl] for _ in range(2)]
    comp = torch.cuda.current_stream()
    ups = [torch.cuda.Stream() for _ in range(n_up)]
    down = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in range(n_up)] for _ in range(2)]  # slot's inputs uploaded
    ev_done = [torch.cuda.Event() for _ in range(2)]  # slot's step computed
    ev_out = [torch.cuda.Event() for _ in range(2)]   # slot's outputs downloaded
    # uploads in chunks of about 32 MB, spread over n_up streams (more than
    # one stream measured no faster: the host link runs at about 180 GB/s)
    chunks = []
    for k, v in host_in.items():
        flat = v.view(-1)
        step_el = max(1, (32 << 20) // v.element_size())
        for a in range(0, flat.numel(), step_el):
            chunks.append((k, a, min(flat.numel(), a + step_el)))

    def upload(i):
        s = i % 2
        for u, st in enumerate(ups):
            with torch.cuda.stream(st):
                if i >= 2:
                    st.wait_event(ev_done[s])  # step i-2 has read this slot's inputs
                for c, (k, a, b) in enumerate(chunks):
                    if c % n_up == u:
                        dev_in[s][k].view(-1)[a:b].copy_(host_in[k].view(-1)[a:b], non_blocking=True)
                ev_in[s][u].record(st)

    def step(i):
        s = i % 2
        for e in ev_in[s]:
            comp.wait_event(e)
        if i >= 2:
            comp.wait_event(ev_out[s])  # step i-2's outputs have been read back
        main.e2e_compute(dev_in[s], dev_out[s])
        ev_done[s].record(comp)
        with torch.cuda.stream(down):
            down.wait_event(ev_done[s])
            for o, h in zip(dev_out[s], host_out[s]):
                h.copy_(o, non_blocking=True)
            ev_out[s].record(down)

    def run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            step(i)
        torch.cuda.synchronize()

    run(warm)
    t0 = time.perf_counter()
    run(steps)
    ms = (time.perf_counter() - t0) * 1e3 / steps
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in tmpl)
    return ms, h2d, d2h


def time_steps(fn, steps, flush, stream):
    """CUDA-event time of each of `steps` calls of fn (L2 flushed between
    calls, outside the timed events).  Returns per-step milliseconds."""
    times = []
    for _ in range(steps):
        if flush is not None:
            flush.add_(1)  # write > L2 bytes
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in times]


# ------------------------------------------------------------------- arms ---


def run_ours(args, ws, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    main = {**WORKLOADS, **PROFILE_ONLY}[args.workload]()
    main.setup(dev)
    # warm-up steps are the timed steps' twins, L2 flush included (the first
    # use of the flush buffer otherwise lands in the first timed step)
    for _ in range(args.warmup):
        flush.add_(1)
        main.run()
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local)
    barrier()
    sampler.start()
    per_step = time_steps(main.run, args.steps, flush, stream)
    barrier()
    clocks = sampler.stop()
    ms, value = aggregate(sum(per_step), args.steps, main.work(),
                          1e12 if main.unit == "TFLOP/s" else 1e9, ws, dev)

    # dominant kernel alone, live CUDA events on its launching stream
    for _ in range(2):
        main.run_dominant()
    dom_ms = statistics.median(time_steps(main.run_dominant, max(3, args.steps), flush, stream))
    peak, peak_src = peak_for(main.bound, long_step=False)
    dom_work = main.dominant_work()
    if main.unit == "TFLOP/s":
        achieved = dom_work / (dom_ms / 1e3) / 1e12
        r_unit = "TFLOP/s"
    else:
        achieved = dom_work / (dom_ms / 1e3) / 1e9
        r_unit = "GB/s"
    roofline = {"bound": main.bound, "achieved": round(achieved, 2),
                "peak": peak, "unit": r_unit,
                "frac": round(achieved / peak, 4) if peak else None,
                "peak_source": peak_src, "traffic": recorded_traffic(main.name),
                "kernel_ms": round(dom_ms, 4)}

    # end-to-end through the public API with host buffers
    e2e = None
    if hasattr(main, "e2e_compute"):
        e_ms, h2d, d2h = run_e2e(main, args.steps)
        e2e = {"value": round(main.scale(e_ms / 1e3) * ws, 3), "unit": main.unit,
               "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h,
               "pipeline": "2 buffer sets; upload, compute and download streams overlap across steps"}
        if hasattr(main, "RESIDENT"):
            e2e["resident_state"] = list(main.RESIDENT)

    rows = {}
    if not args.no_rows:
        for name, cls in WORKLOADS.items():
            if name == main.name:
                continue
            w = cls()
            try:
                w.setup(dev)
                for _ in range(3):
                    w.run()
                t = statistics.median(time_steps(w.run, max(5, args.steps), flush, stream))
                for _ in range(2):
                    w.run_dominant()
                td = statistics.median(time_steps(w.run_dominant, max(5, args.steps), flush, stream))
                pk, src = peak_for(w.bound)
                dw = w.dominant_work() / (td / 1e3) / (1e12 if w.unit == "TFLOP/s" else 1e9)
                rows[name] = {"workload": w.desc, "ms_per_step": round(t, 4),
                              "value": round(w.scale(t / 1e3), 3), "unit": w.unit,
                              "dominant_kernel_ms": round(td, 4),
                              "dominant_achieved": round(dw, 2),
                              "dominant_frac": round(dw / pk, 4) if pk else None,
                              "peak_source": src, "traffic": recorded_traffic(name)}
            except Exception as exc:  # noqa: BLE001
                rows[name] = {"workload": w.desc, "error": str(exc)[:200]}
            del w
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and hasattr(main, "oracle_sample"):
        dt, work, sample = main.oracle_sample()
        cpu = {"value": work / dt / (1e12 if main.unit == "TFLOP/s" else 1e9), "unit": main.unit,
               "cores": torch.get_num_threads(), "kind": "oracle", "sample": sample,
               "seconds": round(dt, 3)}

    if rank == 0:
        line = {
            "metric": "diff-attn fwd TFLOP/s & % BF16 peak (prefill); decode HBM GB/s & % of 8 TB/s",
            "value": round(value, 3), "unit": main.unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": main.dtype, "data": "synthetic",
            "config": {"workload": main.desc, "l2": "flushed between timed steps (512 MB write)",
                       "parallelism": f"replicas x{ws}"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": main.launches * args.steps if main.launches else None,
            "rows": rows, "impl": "ours",
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args, ws, rank):
    """Reference arm: the fp64 CPU oracle, timed as it stands on the host
    cores, on the same bounded sample of the same workload as `cpu_baseline`
    (rank 0 only; other ranks exit without work).  It loads nothing of the
    library: inputs are drawn on the host by `synth` and lambda_init comes
    from the oracle."""
    if rank != 0:
        return
    main = {**WORKLOADS, **PROFILE_ONLY}[args.workload]()
    if not hasattr(main, "oracle_sample"):
        print(json.dumps({"impl": "reference", "unavailable": f"no oracle sample for {main.name}"}))
        return
    main.setup_host()
    for _ in range(args.warmup):
        main.oracle_sample()
    secs, work, sample = 0.0, 0.0, ""
    for _ in range(args.steps):
        dt, w, sample = main.oracle_sample()
        secs += dt
        work += w
    ms = secs * 1e3 / args.steps
    value = work / secs / (1e12 if main.unit == "TFLOP/s" else 1e9)
    line = {"metric": "diff-attn fwd TFLOP/s & % BF16 peak (prefill); decode HBM GB/s & % of 8 TB/s",
            "value": value, "unit": main.unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": main.desc}, "impl": "reference",
            "cpu_baseline": {"value": value, "unit": main.unit, "cores": torch.get_num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": main.unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="v1_fwd", choices=sorted(WORKLOADS) + sorted(PROFILE_ONLY))
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)


if __name__ == "__main__":
    main()
