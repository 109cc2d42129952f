"""GPU parity through the C ABI for the V1 backward (preprocess, tcgen05 main
kernel with 2-CTA clusters, finalize) against the fp64 oracle's chain rule.

Bars (the pages state none for gradients).  The bf16 rounding model
(tests/bf16_model.py: the exact chain rule with only the five bf16 storage
points any bf16 backward has) gives, per input, the error that precision
alone causes; a fixed max-abs bar cannot hold across inputs because that
error grows with the cancellation between the streams (layer 14 at N 129
reaches 11 % of RMS on dV).  So, per gradient tensor:
* max|GPU - oracle| <= k * max|model - oracle| + 1e-3 * RMS(oracle) + floor,
  k = 2 for the backward alone (fed the oracle's forward saves) and k = 3 for
  the training step (GPU forward, then GPU backward on its saves: the
  forward's own bf16 error enters too);
* ||GPU - oracle|| <= max(1.5e-2 ||oracle||, k ||model - oracle||) (2e-2 for
  the step): the second term only matters where a gradient vanishes
  analytically and rounding noise is all that is left;
* dlambda (the lambda-vector gradients are dlambda times fixed vectors)
  within k * the model's error + 2e-3 relative: against the oracle for the
  backward alone; in a training step against the chain rule applied to the
  saves the backward received (dlambda is one sum of <dO, O2> over every row,
  and the forward's own bf16 error in Y, O2 and rstd, which the forward parity
  tests bound, is not part of the rounding model).
floor = 1e-3 * RMS(oracle dV) covers gradients that vanish analytically
(N = 1: dQ, dK and dlambda are exactly zero).
"""

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from bf16_model import bf16, rounded_backward
from oracle import diffattn_oracle as orc

pytestmark = pytest.mark.gpu
BARS = {"bwd": (2.0, 1.5e-2), "step": (3.0, 2e-2)}  # (k, Frobenius)
NAMES = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
GRADS = ("dq1", "dq2", "dk1", "dk2", "dv")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _run(t, li, causal=True, w=None):
    """The training step: GPU forward with saves, then the GPU backward."""
    y, sv = bd.diffattn_v1_fwd(*(t[n] for n in NAMES), li, save=True, causal=causal, rms_weight=w)
    g = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, causal=causal, rms_weight=w)
    torch.cuda.synchronize()
    g["saves"] = dict(t=t, li=li, y=y, sv=sv, w=w)  # what this backward received
    return g


def _dlam_from_saves(sv):
    """dlambda by the chain rule on the saves a backward received (fp64):
    -sum <dO, O2> with dO = c rstd (G - Yhat mean(G Yhat)), Yhat = Y / c; and
    the same with dO rounded to bf16 (the value the kernels hold)."""
    c = 1.0 - sv["li"]
    Y, O2, G = f64(sv["y"]), f64(sv["sv"]["o2"]), f64(sv["t"]["dy"])
    w = 1.0 if sv.get("w") is None else f64(sv["w"])
    rstd = np.transpose(f64(sv["sv"]["rstd"]), (0, 2, 1))[..., None]  # [B, N, H, 1]
    yh = Y / (c * w)
    gw = G * w
    dO = c * rstd * (gw - yh * (gw * yh).mean(-1, keepdims=True))
    return -float(np.sum(dO * O2)), -float(np.sum(bf16(dO) * O2))


def _lam_vectors(t, dlam):
    """The four lambda-vector gradients for a given dlambda (the chain rule
    through lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init)."""
    lq1, lk1, lq2, lk2 = (f64(t[n]) for n in ("lq1", "lk1", "lq2", "lk2"))
    ea, eb = np.exp(lq1 @ lk1), np.exp(lq2 @ lk2)
    return dict(dlq1=dlam * ea * lk1, dlk1=dlam * ea * lq1, dlq2=-dlam * eb * lk2, dlk2=-dlam * eb * lq2)


def _run_exact_saves(t, li, causal=True, w=None):
    """The GPU backward alone, given the oracle's forward outputs."""
    fwd = orc.v1_forward(*(f64(t[n]) for n in NAMES), li, causal=causal,
                         rms_weight=None if w is None else f64(w))
    dev = t["q1"].device
    y = torch.from_numpy(fwd["y"]).to(dev, torch.bfloat16)
    sv = dict(o2=torch.from_numpy(fwd["o2"]).to(dev, torch.bfloat16),
              lse1=torch.from_numpy(fwd["lse1"]).to(dev, torch.float32),
              lse2=torch.from_numpy(fwd["lse2"]).to(dev, torch.float32),
              rstd=torch.from_numpy(fwd["rstd"]).to(dev, torch.float32))
    g = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, causal=causal, rms_weight=w)
    torch.cuda.synchronize()
    return g


def _compare(g, ref, model, heads=None, lam_vectors=True, bar="bwd"):
    k, fro = BARS[bar]
    floor = 1e-3 * float(np.sqrt(np.mean(ref["dv"] ** 2)))
    worst = {}
    for n in GRADS:
        got, exp, mod = f64(g[n]), ref[n], model[n]
        if heads is not None:  # the GPU ran all heads; oracle and model one
            got = got[:, :, heads]
        rms = float(np.sqrt(np.mean(exp ** 2)))
        allowed = k * float(np.max(np.abs(mod - exp))) + 1e-3 * rms + floor
        worst[n] = float(np.max(np.abs(got - exp))) / allowed
        # relative Frobenius bar, or k times the rounding model's own error
        # where the gradient vanishes analytically (N = 1) and only rounding
        # noise is left
        worst[n + "_fro"] = float(np.linalg.norm(got - exp)) / (
            max(fro * float(np.linalg.norm(exp)), k * float(np.linalg.norm(mod - exp)))
            + floor * np.sqrt(exp.size))
    if lam_vectors:
        if "saves" in g:
            # a training step: the backward received the GPU forward's bf16 Y
            # and O2 and its fp32 rstd.  dlambda is a single sum of <dO, O2>
            # over every row, and the forward's own error in those saves
            # (held to its bar by the forward parity tests) can exceed one
            # realisation of the rounding model's; so the lambda-vector
            # gradients are held to the chain rule on the saves received
            dlam_ref, dlam_mod = _dlam_from_saves(g["saves"])
            exp_vec = _lam_vectors(g["saves"]["t"], dlam_ref)
        else:
            dlam_ref, dlam_mod = ref["dlam"], model["dlam"]
            exp_vec = {n: ref[n] for n in ("dlq1", "dlk1", "dlq2", "dlk2")}
        dlam_err = abs(dlam_mod - dlam_ref) / max(abs(dlam_ref), 1e-30)
        for n in ("dlq1", "dlk1", "dlq2", "dlk2"):
            got, exp = f64(g[n]), exp_vec[n]
            scale = float(np.max(np.abs(exp)))
            allowed = (k * dlam_err + 2e-3) * scale + 1e-3 * floor
            worst[n] = float(np.max(np.abs(got - exp))) / allowed
    assert max(worst.values()) <= 1.0, worst


def _model(t, li, heads=None, causal=True, w=None):
    f = {n: f64(t[n]) for n in NAMES + ("dy",)}
    wf = None if w is None else f64(w)
    fwd = orc.v1_forward(*(f[n] for n in NAMES), li, causal=causal, rms_weight=wf)
    return rounded_backward(f, fwd, li, heads=heads, causal=causal, rms_weight=wf)


@pytest.mark.parametrize("B,N,H,layer", [(1, 200, 2, 1), (2, 384, 1, 3), (1, 129, 2, 14),
                                          (1, 1, 1, 1), (1, 700, 3, 28), (2, 7, 2, 2), (1, 64, 2, 5)])
def test_v1_bwd_parity_small(B, N, H, layer):
    t = synth.v1_inputs(B, N, H, 128, 256, "bf16", seed=5000 + N + H, device="cuda", with_dy=True)
    li = float(np.float32(bd.diffattn_lambda_init(layer)))
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]))
    model = _model(t, li)
    _compare(_run_exact_saves(t, li), ref, model, bar="bwd")
    _compare(_run(t, li), ref, model, bar="step")


@pytest.mark.parametrize("B,N,H,layer", [(1, 200, 2, 1), (2, 129, 1, 14), (1, 1, 1, 1), (1, 500, 2, 5)])
def test_v1_bwd_parity_head_dims_64_128(B, N, H, layer):
    """Head dims (64, 128): half-width K, Q tiles, one dQ^T half (feature rows
    64-127 are zero padding), dV halves of 64 columns exchanged."""
    t = synth.v1_inputs(B, N, H, 64, 128, "bf16", seed=5100 + N + H, device="cuda", with_dy=True)
    li = float(np.float32(bd.diffattn_lambda_init(layer)))
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]))
    model = _model(t, li)
    _compare(_run_exact_saves(t, li), ref, model, bar="bwd")
    _compare(_run(t, li), ref, model, bar="step")


def test_v1_bwd_deterministic_head_dims_64_128():
    """Deterministic dQ slots at head dims (64, 128): a bitwise repeat; dK, dV
    and the lambda-vector gradients bitwise equal to the default mode's (the
    mode changes only how dQ leaves the main kernel); dQ, dK, dV against the
    oracle.  (The lambda-vector gradients' oracle bar is checked by the
    backward-alone parity tests: in a training step dlambda sums <dO, O2> over
    every row of the bf16 forward outputs, whose own error the rounding model
    does not count.)"""
    t = synth.v1_inputs(1, 400, 2, 64, 128, "bf16", seed=5150, device="cuda", with_dy=True)
    li = float(np.float32(bd.diffattn_lambda_init(3)))
    y, sv = bd.diffattn_v1_fwd(*(t[n] for n in NAMES), li, save=True)
    g0 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv)
    g1 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, deterministic=True)
    g2 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, deterministic=True)
    torch.cuda.synchronize()
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n
    for n in ("dk1", "dk2", "dv", "dlq1", "dlk1", "dlq2", "dlk2"):
        assert torch.equal(g0[n], g1[n]), n
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]))
    _compare(g1, ref, _model(t, li), lam_vectors=False, bar="step")


@pytest.mark.parametrize("B,N,H,dqk,layer", [(1, 200, 2, 128, 1), (2, 129, 1, 64, 14), (1, 1, 1, 128, 1),
                                              (1, 300, 2, 128, 5)])
def test_v1_bwd_parity_not_causal(B, N, H, dqk, layer):
    """Every key attends every query: each key tile walks all query tiles,
    no diagonal mask; ragged key tails (zero K and V rows past N)."""
    t = synth.v1_inputs(B, N, H, dqk, 2 * dqk, "bf16", seed=5200 + N + H, device="cuda", with_dy=True)
    li = float(np.float32(bd.diffattn_lambda_init(layer)))
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]), causal=False)
    model = _model(t, li, causal=False)
    _compare(_run_exact_saves(t, li, causal=False), ref, model, bar="bwd")
    _compare(_run(t, li, causal=False), ref, model, bar="step")


@pytest.mark.parametrize("B,N,H,dqk,layer", [(1, 200, 2, 128, 1), (2, 129, 1, 64, 14)])
def test_v1_bwd_parity_rms_weight(B, N, H, dqk, layer):
    """A non-unit RMSNorm weight w (fixed: no gradient): the preprocess takes
    the normalised output as Y / ((1 - lambda_init) w) and dOhat = c w G."""
    t = synth.v1_inputs(B, N, H, dqk, 2 * dqk, "bf16", seed=5300 + N + H, device="cuda", with_dy=True)
    w = 0.5 + torch.rand(2 * dqk, generator=torch.Generator().manual_seed(5301), dtype=torch.float32).cuda()
    li = float(np.float32(bd.diffattn_lambda_init(layer)))
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]), rms_weight=f64(w))
    model = _model(t, li, w=w)
    _compare(_run_exact_saves(t, li, w=w), ref, model, bar="bwd")
    _compare(_run(t, li, w=w), ref, model, bar="step")


def test_v1_bwd_strided_packed_views():
    """q1/q2 and k1/k2 as views into packed [B, N, H, 2, d_qk] buffers, and the
    gradients written into views of packed buffers of the same layout: the
    backward equals the one on contiguous copies bit for bit."""
    B, N, H = 1, 260, 2
    t = synth.v1_inputs(B, N, H, 128, 256, "bf16", seed=5400, device="cuda", with_dy=True)
    qp = torch.stack([t["q1"], t["q2"]], dim=3).contiguous()
    kp = torch.stack([t["k1"], t["k2"]], dim=3).contiguous()
    tv = dict(t, q1=qp[:, :, :, 0], q2=qp[:, :, :, 1], k1=kp[:, :, :, 0], k2=kp[:, :, :, 1])
    li = float(np.float32(bd.diffattn_lambda_init(2)))
    y, sv = bd.diffattn_v1_fwd(*(t[n] for n in NAMES), li, save=True)
    ref = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv)
    dqp = torch.empty_like(qp)
    dkp = torch.empty_like(kp)
    grads = dict(dq1=dqp[:, :, :, 0], dq2=dqp[:, :, :, 1], dk1=dkp[:, :, :, 0], dk2=dkp[:, :, :, 1],
                 dv=torch.empty_like(t["v"]), dlq1=torch.empty_like(t["lq1"]), dlk1=torch.empty_like(t["lk1"]),
                 dlq2=torch.empty_like(t["lq2"]), dlk2=torch.empty_like(t["lk2"]))
    got = bd.diffattn_v1_bwd(*(tv[n] for n in NAMES), li, y, t["dy"], sv, grads=grads)
    torch.cuda.synchronize()
    for n in ("dk1", "dk2", "dv", "dlq1", "dlk1", "dlq2", "dlk2"):
        assert torch.equal(got[n], ref[n]), n
    for n in ("dq1", "dq2"):  # fp32 reduce-adds: order may differ run to run
        assert torch.allclose(got[n].float(), ref[n].float(), rtol=1e-2, atol=1e-3 * float(ref[n].float().abs().max()))


def test_v1_bwd_deterministic_parts_repeat():
    """dK and dV come from one CTA each (no atomics): bitwise equal on a rerun."""
    t = synth.v1_inputs(1, 300, 2, 128, 256, "bf16", seed=61, device="cuda", with_dy=True)
    li = bd.diffattn_lambda_init(2)
    g1 = _run(t, li)
    g2 = _run(t, li)
    for n in ("dk1", "dk2", "dv"):
        assert torch.equal(g1[n], g2[n]), n


def test_v1_bwd_h16_n1024_all_heads():
    """16 heads at N 1024: every gradient incl. the lambda vectors (dlambda
    sums over all heads and rows)."""
    t = synth.v1_inputs(1, 1024, 16, 128, 256, "bf16", seed=62, device="cuda", with_dy=True)
    li = float(np.float32(bd.diffattn_lambda_init(1)))
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]))
    model = _model(t, li)
    _compare(_run_exact_saves(t, li), ref, model, bar="bwd")
    _compare(_run(t, li), ref, model, bar="step")


def test_v1_bwd_full_size_b1_h16_n8192_one_head():
    """B1 H16 N8192 (the training-step workload) through the library; the
    oracle recomputes one head completely (its lambda-vector gradients are
    partial, so only dQ, dK, dV are compared)."""
    t = synth.v1_inputs(1, 8192, 16, 128, 256, "bf16", seed=1005, device="cuda", with_dy=True)
    li = bd.diffattn_lambda_init(1)
    g = _run(t, li)
    h = 5
    li = float(np.float32(li))
    th = {n: (t[n][:, :, h:h + 1] if t[n].dim() == 4 else t[n]) for n in NAMES + ("dy",)}
    ref = orc.v1_backward(*(f64(th[n]) for n in NAMES), li, f64(th["dy"]))
    model = _model(th, li)
    _compare(g, ref, model, heads=slice(h, h + 1), lam_vectors=False, bar="step")


@pytest.mark.parametrize("B,N,H,layer", [(1, 300, 2, 2), (2, 129, 1, 14), (1, 1, 1, 1)])
def test_v1_bwd_deterministic_mode(B, N, H, layer):
    """deterministic=True: dQ from per-key-tile slots summed in a fixed order.
    Same bars as the default mode, and bitwise equal results on a rerun."""
    t = synth.v1_inputs(B, N, H, 128, 256, "bf16", seed=5100 + N + H, device="cuda", with_dy=True)
    li = float(np.float32(bd.diffattn_lambda_init(layer)))
    ref = orc.v1_backward(*(f64(t[n]) for n in NAMES), li, f64(t["dy"]))
    model = _model(t, li)
    y, sv = bd.diffattn_v1_fwd(*(t[n] for n in NAMES), li, save=True)
    g1 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, deterministic=True)
    g2 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, deterministic=True)
    torch.cuda.synchronize()
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n
    g1["saves"] = dict(t=t, li=li, y=y, sv=sv)
    _compare(g1, ref, model, bar="step")


def test_v1_bwd_deterministic_full_size_repeat():
    """B1 H16 N8192: two deterministic backward runs agree bit for bit, and
    agree with the default (reduce-add) mode to within bf16 rounding."""
    t = synth.v1_inputs(1, 8192, 16, 128, 256, "bf16", seed=1005, device="cuda", with_dy=True)
    li = bd.diffattn_lambda_init(1)
    y, sv = bd.diffattn_v1_fwd(*(t[n] for n in NAMES), li, save=True)
    g1 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, deterministic=True)
    g2 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv, deterministic=True)
    g3 = bd.diffattn_v1_bwd(*(t[n] for n in NAMES), li, y, t["dy"], sv)
    torch.cuda.synchronize()
    for n in g1:
        assert torch.equal(g1[n], g2[n]), n
    for n in ("dq1", "dq2"):
        a, b = g1[n].float(), g3[n].float()
        rms = float(a.pow(2).mean().sqrt())
        assert float((a - b).abs().max()) <= 2e-2 * rms, n
    for n in ("dk1", "dk2", "dv"):
        assert torch.equal(g1[n], g3[n]), n
