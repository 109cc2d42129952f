"""Where the V1 backward's tolerance comes from (CPU, no GPU).

The library's backward stores Y and O2 (forward outputs) in bf16, feeds dO
to the tensor cores in bf16 and writes P and dS in bf16 as MMA operands, as
any bf16 attention backward must.  tests/bf16_model.py runs the backward in
exact fp64 EXCEPT for those five bf16 roundings and measures the error
against the fp64 oracle.  This test documents two facts the GPU bars rest on:

* the rounding model alone exceeds a fixed 2e-2 * RMS max-abs bar (so no
  fixed max-abs bar of that size can hold for a bf16 backward: the tail
  grows with the cancellation between the two streams), while
* its Frobenius error stays well under 1.5e-2.

The GPU tests therefore bound the library's max error by a small multiple of
the model's error on the same inputs, and its Frobenius error by a fixed bar.
"""

import numpy as np
import torch

from differential_attention_diff_gb300 import synth
from bf16_model import (rounded_backward, rounded_backward_grouped, rounded_backward_v2, rounded_forward,
                        rounded_grouped_forward)
from oracle import diffattn_oracle as orc


def test_bf16_rounding_model_sets_the_gradient_tolerance():
    t = synth.v1_inputs(1, 200, 2, 128, 256, "bf16", seed=5202, device="cpu", with_dy=True)
    f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    li = float(np.float32(orc.lambda_init(1)))
    names = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
    ref = orc.v1_backward(*(f[n] for n in names), li, f["dy"])
    fwd = orc.v1_forward(*(f[n] for n in names), li)
    got = rounded_backward(f, fwd, li)
    maxrel, fro = {}, {}
    for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
        e = ref[n]
        maxrel[n] = float(np.max(np.abs(got[n] - e)) / np.sqrt(np.mean(e ** 2)))
        fro[n] = float(np.linalg.norm(got[n] - e) / np.linalg.norm(e))
    assert max(maxrel.values()) > 2e-2, maxrel     # a fixed 2e-2 bar is unreachable
    assert max(fro.values()) < 0.5 * 1.5e-2, fro   # the Frobenius bar leaves margin


def test_v2_rounding_model_is_the_chain_rule_and_sets_the_tolerance():
    """The V2 model without rounding reproduces the oracle's gradients (so it
    rounds the right quantities of the right formula); with bf16 rounding its
    Frobenius error stays well under the GPU bars."""
    t = synth.v2_inputs(1, 150, 2, 1, 128, 64, seed=5203, device="cpu", with_dout=True)
    f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    ref = orc.v2_backward(f["q"], f["k"], f["v"], f["x"], f["w_lambda"], f["dout"])
    fwd = orc.v2_forward(f["q"], f["k"], f["v"], ref["gate"])
    exact = rounded_backward_v2(f, fwd, ref["gate"], rnd=lambda a: a)
    for n in ("dq", "dk", "dv", "dz", "dx", "dw"):
        np.testing.assert_allclose(exact[n], ref[n], rtol=1e-10, atol=1e-12 * np.abs(ref[n]).max())
    got = rounded_backward_v2(f, fwd, ref["gate"])
    for n in ("dq", "dk", "dv", "dz", "dx", "dw"):
        fro = float(np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n]))
        assert fro < 0.5 * 1.5e-2, (n, fro)


def test_grouped_rounding_model_is_the_chain_rule_and_sets_the_tolerance():
    """The grouped model without rounding reproduces the oracle's grouped
    backward (it rounds the right quantities of the right formula), equals the
    V2 model at ratio 1, and with bf16 rounding keeps its Frobenius error well
    under the GPU bars."""
    t = synth.grouped_inputs(1, 150, 6, 3, 1, 64, 64, seed=5204, device="cpu")
    t["dout"] = torch.randn((1, 150, 6, 64), generator=torch.Generator().manual_seed(5205)).to(torch.bfloat16)
    f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    ref = orc.grouped_backward(f["q"], f["k"], f["v"], f["x"], f["w_lambda"], f["dout"], 3)
    fwd = orc.grouped_forward(f["q"], f["k"], f["v"], ref["gate"], 3)
    exact = rounded_backward_grouped(f, fwd, ref["gate"], 3, rnd=lambda a: a)
    for n in ("dq", "dk", "dv", "dz", "dx", "dw"):
        np.testing.assert_allclose(exact[n], ref[n], rtol=1e-10, atol=1e-12 * np.abs(ref[n]).max())
    got = rounded_backward_grouped(f, fwd, ref["gate"], 3)
    for n in ("dq", "dk", "dv", "dz", "dx", "dw"):
        fro = float(np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n]))
        assert fro < 0.5 * 1.5e-2, (n, fro)
    t2 = synth.v2_inputs(1, 70, 2, 1, 64, 64, seed=5206, device="cpu", with_dout=True)
    f2 = {k: v.to(torch.float64).numpy() for k, v in t2.items()}
    ref2 = orc.v2_backward(f2["q"], f2["k"], f2["v"], f2["x"], f2["w_lambda"], f2["dout"])
    fwd2 = orc.v2_forward(f2["q"], f2["k"], f2["v"], ref2["gate"])
    a = rounded_backward_grouped(f2, fwd2, ref2["gate"], 1)
    b = rounded_backward_v2(f2, fwd2, ref2["gate"])
    for n in ("dq", "dk", "dv", "dz", "dx", "dw"):
        np.testing.assert_allclose(a[n], b[n], rtol=1e-12, atol=1e-12 * np.abs(b[n]).max())


def test_v1_forward_rounding_model_and_the_step_bar():
    """The V1 forward model behind the training step's bar.  Without rounding
    it reproduces the oracle forward (Y, O2, rstd), so it rounds the right
    quantities of the right formula.  With its bf16 points, the forward's Y
    error stays inside the forward tests' 2e-2 * RMS(V).  Under strong
    cancellation between the streams (lambda vectors chosen so that
    lambda = 1 at layer 13: O1 - O2 is small in long rows, and rstd large),
    the backward fed the rounded forward has several times the dQ/dK error
    of the backward fed exact forward outputs.  That is why the step's
    max-abs bar takes the forward-aware model.  Its Frobenius error stays
    well under the step's fixed 2e-2 bar."""
    names = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
    t = synth.v1_inputs(1, 256, 2, 64, 128, "bf16", seed=5221, device="cpu", with_dy=True)
    f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    li = float(np.float32(orc.lambda_init(13)))
    # lambda = exp(lq1.lk1) - exp(lq2.lk2) + lambda_init = 1
    e0 = np.zeros(64)
    e0[0] = np.sqrt(np.log(2.0 - li))
    f["lq1"] = f["lk1"] = e0
    f["lq2"] = f["lk2"] = np.zeros(64)
    fwd = orc.v1_forward(*(f[n] for n in names), li)
    assert abs(fwd["lam"] - 1.0) < 1e-12
    exact = rounded_forward(f, fwd, li, rnd=lambda a: a)
    np.testing.assert_allclose(exact["y"], fwd["y"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(exact["o2"], fwd["o2"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(exact["rstd"], fwd["rstd"], rtol=1e-12)
    rf = rounded_forward(f, fwd, li)
    rms_v = float(np.sqrt(np.mean(f["v"] ** 2)))
    assert np.max(np.abs(rf["y"] - fwd["y"])) <= 2e-2 * rms_v
    ref = orc.v1_backward(*(f[n] for n in names), li, f["dy"])
    bwd_only = rounded_backward(f, fwd, li)
    step = rounded_backward(f, rf, li)
    grow = max(np.max(np.abs(step[n] - ref[n])) / np.max(np.abs(bwd_only[n] - ref[n]))
               for n in ("dq1", "dq2", "dk1", "dk2"))
    assert grow > 2.0, grow
    for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
        assert np.linalg.norm(step[n] - ref[n]) / np.linalg.norm(ref[n]) < 0.5 * 2e-2, n


def test_v1_rounding_model_is_the_chain_rule():
    """The V1 backward model with its rounding switched off reproduces the
    oracle's gradients and dlambda (causal or not, with an RMSNorm weight), so
    it rounds the right quantities of the right formula; the per-row dlambda
    error it reports is then zero."""
    names = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
    t = synth.v1_inputs(2, 70, 2, 64, 128, "bf16", seed=5240, device="cpu", with_dy=True)
    f = {k: v.to(torch.float64).numpy() for k, v in t.items()}
    li = float(np.float32(orc.lambda_init(5)))
    w = 0.5 + np.arange(128) / 256.0
    for causal in (True, False):
        ref = orc.v1_backward(*(f[n] for n in names), li, f["dy"], causal=causal, rms_weight=w)
        fwd = orc.v1_forward(*(f[n] for n in names), li, causal=causal, rms_weight=w)
        exact = rounded_backward(f, fwd, li, causal=causal, rms_weight=w, rnd=lambda a: a, exact_fwd=fwd)
        for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
            np.testing.assert_allclose(exact[n], ref[n], rtol=0, atol=1e-12 * np.abs(ref[n]).max())
        assert abs(exact["dlam"] - ref["dlam"]) <= 1e-12 * abs(ref["dlam"])
        assert exact["dlam_ss"] == 0.0


def test_grouped_forward_rounding_model_is_the_forward():
    """The grouped forward model with its rounding switched off is the
    oracle's grouped forward (causal or not, a non-default scale); with bf16
    rounding it stays inside the 2e-2 * RMS(V) output bar on ordinary inputs."""
    rng = np.random.default_rng(5250)
    N, r, d = 60, 3, 64
    q = rng.standard_normal((N, r + 1, d))
    k = rng.standard_normal((N, d))
    v = rng.standard_normal((N, d))
    g = rng.uniform(0.0, 1.0, (N, r))
    for causal in (True, False):
        ref = orc.grouped_forward(q[None], k[None, :, None], v[None, :, None], g[None], r, causal=causal,
                                  scale=0.1)["out"][0]
        exact = rounded_grouped_forward(q, k, v, g, r, scale=0.1, causal=causal, rnd=lambda a: a)
        np.testing.assert_allclose(exact, ref, rtol=0, atol=1e-12)
        rounded = rounded_grouped_forward(q, k, v, g, r, scale=0.1, causal=causal)
        assert np.max(np.abs(rounded - ref)) <= 2e-2 * np.sqrt(np.mean(v ** 2))
