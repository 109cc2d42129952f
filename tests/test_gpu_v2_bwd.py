"""GPU parity through the C ABI for the V2 backward (preprocess, tcgen05 main
kernel, finalize, gate-projection gradients) against the fp64 oracle's chain
rule.

Bars, as for the V1 backward (the pages state none for gradients): the bf16
rounding model (tests/bf16_model.py, rounded_backward_v2: the exact chain
rule with only the bf16 storage points any bf16 backward has) gives the error
precision alone causes on the same inputs.  Per gradient tensor:
* max|GPU - oracle| <= k * max|model - oracle| + 1e-3 * RMS(oracle) + floor,
  k = 2 for the backward alone (fed the oracle's forward saves), 3 for the
  training step (GPU forward with saves, then the GPU backward);
* ||GPU - oracle|| <= 1.5e-2 ||oracle|| (2e-2 for the step), a fixed bar that
  does not involve the model; only where a gradient vanishes analytically
  (N = 1: dQ and dK are exactly zero, the oracle's norm is rounding residue)
  is it k times the model's own Frobenius error;
floor = 1e-3 * RMS(oracle dV) for dQ / dK / dV and 1e-3 * RMS of the tensor
itself for the gate gradients.  Every expected value is the oracle's.  Each
test records error / allowed per tensor (tests/ratio_log.py).
"""

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from bf16_model import rounded_backward_v2
from oracle import diffattn_oracle as orc
from ratio_log import record

pytestmark = pytest.mark.gpu
BARS = {"bwd": (2.0, 1.5e-2), "step": (3.0, 2e-2)}
ATTN = ("dq", "dk", "dv")
GATE = ("dz", "dx", "dw")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _run(t, causal=True, scale=None):
    """The training step: GPU forward with saves, then the GPU backward
    (scale: the softmax scale, None = the default 1/sqrt(d))."""
    ss = 0.0 if scale is None else scale
    _, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True,
                               causal=causal, softmax_scale=ss)
    g = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"],
                           want_dz=True, causal=causal, softmax_scale=ss)
    torch.cuda.synchronize()
    return g


def _run_exact_saves(t, fwd, causal=True, scale=None):
    """The GPU backward alone, given the oracle's forward saves."""
    dev = t["q"].device
    sv = dict(o_heads=torch.from_numpy(fwd["o"]).to(dev, torch.bfloat16),
              lse=torch.from_numpy(fwd["lse"]).to(dev, torch.float32))
    g = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"],
                           want_dz=True, causal=causal, softmax_scale=0.0 if scale is None else scale)
    torch.cuda.synchronize()
    return g


def _reference(t, causal=True, scale=None):
    f = {n: f64(v) for n, v in t.items()}
    ref = orc.v2_backward(f["q"], f["k"], f["v"], f["x"], f["w_lambda"], f["dout"], causal=causal, scale=scale)
    fwd = dict(o=ref["o"], lse=ref["lse"])  # the forward the oracle's chain rule ran on
    model = rounded_backward_v2(f, fwd, ref["gate"], causal=causal, scale=scale)
    return ref, fwd, model


def _compare(g, ref, model, names=ATTN + GATE, bar="bwd", sl=None):
    k, fro = BARS[bar]
    floor_attn = 1e-3 * float(np.sqrt(np.mean(ref["dv"] ** 2)))
    dv_norm = float(np.linalg.norm(ref["dv"]))
    worst = {}
    for n in names:
        got, exp, mod = f64(g[n]), ref[n], model[n]
        if sl is not None and n in sl:  # the GPU ran every head; oracle and model a slice
            got = got[sl[n]]
        rms = float(np.sqrt(np.mean(exp ** 2)))
        floor = floor_attn if n in ATTN else 1e-3 * rms
        allowed = k * float(np.max(np.abs(mod - exp))) + 1e-3 * rms + floor
        worst[n] = float(np.max(np.abs(got - exp))) / allowed
        exp_norm = float(np.linalg.norm(exp))
        if exp_norm > 1e-9 * dv_norm:
            fro_allowed = fro * exp_norm
        else:  # analytically zero (N = 1): rounding noise against rounding noise
            fro_allowed = k * float(np.linalg.norm(mod - exp))
        worst[n + "_fro"] = float(np.linalg.norm(got - exp)) / (fro_allowed + floor * np.sqrt(exp.size))
    record(worst, bar)
    assert max(worst.values()) <= 1.0, worst


@pytest.mark.parametrize("B,N,h,hkv", [(1, 200, 2, 1), (2, 129, 2, 2), (1, 1, 1, 1), (1, 300, 4, 1),
                                        (1, 700, 4, 2), (2, 64, 8, 2), (2, 7, 2, 1)])
def test_v2_bwd_parity_small(B, N, h, hkv):
    """Query-head groups of 2, 4 and 8, one token, ragged tails across several
    128-key tiles, two batches."""
    t = synth.v2_inputs(B, N, h, hkv, 128, 128, seed=7000 + N + h, device="cuda", with_dout=True)
    ref, fwd, model = _reference(t)
    _compare(_run_exact_saves(t, fwd), ref, model, bar="bwd")
    _compare(_run(t), ref, model, bar="step")


@pytest.mark.parametrize("B,N,h,hkv", [(1, 200, 2, 1), (2, 129, 2, 2), (1, 1, 1, 1), (1, 300, 4, 1)])
def test_v2_bwd_parity_head_dim_64(B, N, h, hkv):
    """Head dim 64: half-width K, V, Q and dO tiles, dV and dK in 64 TMEM
    columns, dQ^T with 64 zero feature rows that are never stored."""
    t = synth.v2_inputs(B, N, h, hkv, 64, 128, seed=7200 + N + h, device="cuda", with_dout=True)
    ref, fwd, model = _reference(t)
    _compare(_run_exact_saves(t, fwd), ref, model, bar="bwd")
    _compare(_run(t), ref, model, bar="step")


@pytest.mark.parametrize("B,N,h,hkv,d", [(1, 200, 2, 1, 128), (2, 129, 2, 2, 64), (1, 1, 1, 1, 128),
                                          (1, 300, 4, 1, 128)])
def test_v2_bwd_parity_not_causal(B, N, h, hkv, d):
    """Every key attends every query: each key tile walks all query tiles of
    every head, no diagonal mask; ragged key tails."""
    t = synth.v2_inputs(B, N, h, hkv, d, 128, seed=7300 + N + h, device="cuda", with_dout=True)
    ref, fwd, model = _reference(t, causal=False)
    _compare(_run_exact_saves(t, fwd, causal=False), ref, model, bar="bwd")
    _compare(_run(t, causal=False), ref, model, bar="step")


def test_v2_bwd_strided_views():
    """q, k, v as views into one packed [B, N, 2h + 2 h_kv, d] buffer: the
    backward equals the one on contiguous copies (dK, dV bit for bit)."""
    B, N, h, hkv = 1, 300, 4, 2
    t = synth.v2_inputs(B, N, h, hkv, 128, 128, seed=7400, device="cuda", with_dout=True)
    buf = torch.cat([t["q"], t["k"], t["v"]], dim=2).contiguous()
    tv = dict(t, q=buf[:, :, :2 * h], k=buf[:, :, 2 * h:2 * h + hkv], v=buf[:, :, 2 * h + hkv:])
    _, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True)
    ref = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"])
    got = bd.diffattn_v2_bwd(tv["q"], tv["k"], tv["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    for n in ("dk", "dv"):
        assert torch.equal(got[n], ref[n]), n
    assert torch.allclose(got["dq"].float(), ref["dq"].float(), rtol=1e-2,
                          atol=1e-3 * float(ref["dq"].float().abs().max()))


def test_v2_bwd_gate_given_matches_gate_from_x():
    """A caller-supplied gate (the same values) gives the same dQ, dK, dV as
    the gate computed from x and W inside the call."""
    t = synth.v2_inputs(1, 260, 2, 1, 128, 128, seed=7101, device="cuda", with_dout=True)
    _, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True)
    gate = bd.diffattn_v2_gate(t["x"], t["w_lambda"])
    g1 = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"])
    g2 = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, gate=gate)
    torch.cuda.synchronize()
    assert set(g2) == {"dq", "dk", "dv"}
    for n in ("dk", "dv"):
        assert torch.equal(g1[n], g2[n]), n
    assert torch.allclose(g1["dq"].float(), g2["dq"].float(), rtol=1e-2, atol=1e-3)


def test_v2_bwd_deterministic_parts_repeat():
    """dK, dV (one CTA each, no atomics) and the gate gradients (fixed-order
    reductions) are bitwise equal on a rerun."""
    t = synth.v2_inputs(1, 400, 4, 1, 128, 128, seed=7102, device="cuda", with_dout=True)
    g1 = _run(t)
    g2 = _run(t)
    for n in ("dk", "dv", "dz", "dx", "dw"):
        assert torch.equal(g1[n], g2[n]), n


def test_v2_bwd_zero_gate_weight_odd_heads_get_half_gradient():
    """W_lambda = 0 makes every gate 1/2: the odd heads' dO is exactly -G/2,
    so with q_odd = q_even the odd heads' dQ is -1/2 of the even heads' (the
    bf16 rounding of -G/2 is exact)."""
    t = synth.v2_inputs(1, 300, 2, 1, 128, 128, seed=7103, device="cuda", with_dout=True)
    t["w_lambda"].zero_()
    t["q"][:, :, 1::2] = t["q"][:, :, 0::2]
    g = _run(t)
    ev, od = g["dq"][:, :, 0::2].float(), g["dq"][:, :, 1::2].float()
    assert torch.allclose(od, -0.5 * ev, rtol=2e-2, atol=1e-3 * float(ev.abs().max()))


def test_v2_bwd_full_size_b2_n8192_64q_8kv_one_group():
    """B2 N8192, 64 query heads over 8 K/V heads, d_model 4096 (the V2 prefill
    workload) through the library; the oracle recomputes one (batch, K/V
    group) completely: its 8 query heads' dQ, the group's dK and dV, and dz
    of its 4 pairs."""
    t = synth.v2_inputs(2, 8192, 32, 8, 128, 4096, seed=1003, device="cuda", with_dout=True)
    g = _run(t)
    b, grp = 1, 5
    qs, ps = slice(8 * grp, 8 * grp + 8), slice(4 * grp, 4 * grp + 4)
    ts = dict(q=t["q"][b:b + 1, :, qs], k=t["k"][b:b + 1, :, grp:grp + 1], v=t["v"][b:b + 1, :, grp:grp + 1],
              x=t["x"][b:b + 1], w_lambda=t["w_lambda"][:, ps], dout=t["dout"][b:b + 1, :, ps])
    ref, _, model = _reference(ts)
    sl = dict(dq=(slice(b, b + 1), slice(None), qs), dk=(slice(b, b + 1), slice(None), slice(grp, grp + 1)),
              dv=(slice(b, b + 1), slice(None), slice(grp, grp + 1)), dz=(slice(b, b + 1), slice(None), ps))
    _compare(g, ref, model, names=ATTN + ("dz",), bar="step", sl=sl)


@pytest.mark.parametrize("B,N,h,dm", [(2, 200, 8, 320), (1, 300, 16, 128), (1, 129, 24, 256),
                                      (2, 160, 32, 384), (1, 257, 64, 512), (1, 1100, 32, 256)])
def test_v2_bwd_gate_grads_are_products(B, N, h, dm):
    """dX = dz W^T and dW = X^T dz, checked against the products of the
    call's own dz (fp64) with W and X: bars independent of the attention's
    error.  The shapes reach the tensor-core kernels (T >= 128, h % 8 == 0;
    dW also d_model % 128 == 0, else its CUDA-core kernel) with a ragged last
    token block, a partial last 256-feature tile of dX (d_model 320 / 384),
    h from 8 to 64 gate heads and, at T = 1100, two 1024-token dW chunks."""
    t = synth.v2_inputs(B, N, h, 1, 128, dm, seed=7500 + h + dm, device="cuda", with_dout=True)
    _, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True)
    g = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"], want_dz=True)
    torch.cuda.synchronize()
    dz = f64(g["dz"]).reshape(B * N, h)
    # dX in bf16: one rounding of a product carried to about 16 bits, so
    # within one bf16 ulp of the exact value
    ref = dz @ f64(t["w_lambda"]).T
    got = f64(g["dx"]).reshape(B * N, dm)
    ref_bf16 = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    tol = np.abs(ref) * 2.0 ** -7 + 1e-6 * float(np.abs(ref).max())
    assert np.all(np.abs(got - ref_bf16) <= tol), float((np.abs(got - ref_bf16) / tol).max())
    # dW in fp32, summed over the tokens
    ref_w = f64(t["x"]).reshape(B * N, dm).T @ dz
    got_w = f64(g["dw"])
    tol_w = 1e-3 * np.abs(ref_w) + 1e-4 * float(np.abs(ref_w).max())
    assert np.all(np.abs(got_w - ref_w) <= tol_w), float((np.abs(got_w - ref_w) / tol_w).max())
