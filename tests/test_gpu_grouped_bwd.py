"""GPU parity through the C ABI for the grouped differential attention
backward (the grouped preprocess, then the V2 backward's tcgen05 main kernel,
finalize and gate-projection gradients) against the fp64 oracle's chain rule
(orc.grouped_backward).

Bars, as for the V2 backward (the pages state none for gradients): the bf16
rounding model (tests/bf16_model.py, rounded_backward_grouped: the exact
chain rule with only the bf16 storage points any bf16 backward has, the
noise heads' dO = -sum_i g_i dOut_i among them) gives the error precision
alone causes on the same inputs.  Per gradient tensor:
* max|GPU - oracle| <= k * max|model - oracle| + 1e-3 * RMS(oracle) + floor,
  k = 2 for the backward alone (fed the oracle's forward saves), 3 for the
  training step (GPU grouped forward with saves, then the GPU backward);
* ||GPU - oracle|| <= 1.5e-2 ||oracle|| (2e-2 for the step); where a gradient
  vanishes analytically (N = 1: dQ and dK) k times the model's own error;
floor = 1e-3 * RMS(oracle dV) for dQ / dK / dV and 1e-3 * RMS of the tensor
itself for the gate gradients.  Each test records error / allowed per tensor
(tests/ratio_log.py).
"""

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from bf16_model import rounded_backward_grouped
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


def _inputs(B, N, h, ratio, hkv, d, dm, seed):
    t = synth.grouped_inputs(B, N, h, ratio, hkv, d, dm, seed=seed, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    t["dout"] = torch.randn((B, N, h, d), generator=g, device="cuda").to(torch.bfloat16)
    return t


def _forward_saves(t, ratio, causal=True, scale=None):
    B, N, Hq, d = t["q"].shape
    heads = torch.empty((B, N, Hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, Hq, N), dtype=torch.float32, device="cuda")
    bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], ratio, x=t["x"], w_lambda=t["w_lambda"], o_heads=heads,
                            lse=lse, causal=causal, softmax_scale=0.0 if scale is None else scale)
    return dict(o_heads=heads, lse=lse)


def _run(t, ratio, causal=True, scale=None):
    """The training step: GPU grouped forward with saves, then the backward."""
    sv = _forward_saves(t, ratio, causal, scale)
    g = bd.diffattn_grouped_bwd(t["q"], t["k"], t["v"], t["dout"], sv, ratio, x=t["x"], w_lambda=t["w_lambda"],
                                want_dz=True, causal=causal, softmax_scale=0.0 if scale is None else scale)
    torch.cuda.synchronize()
    return g


def _run_exact_saves(t, ratio, ref, causal=True, scale=None):
    """The GPU backward alone, given the oracle's forward saves."""
    sv = dict(o_heads=torch.from_numpy(ref["o"]).to("cuda", torch.bfloat16),
              lse=torch.from_numpy(ref["lse"]).to("cuda", torch.float32))
    g = bd.diffattn_grouped_bwd(t["q"], t["k"], t["v"], t["dout"], sv, ratio, x=t["x"], w_lambda=t["w_lambda"],
                                want_dz=True, causal=causal, softmax_scale=0.0 if scale is None else scale)
    torch.cuda.synchronize()
    return g


def _reference(t, ratio, causal=True, scale=None):
    f = {n: f64(v) for n, v in t.items()}
    ref = orc.grouped_backward(f["q"], f["k"], f["v"], f["x"], f["w_lambda"], f["dout"], ratio, causal=causal,
                               scale=scale)
    fwd = dict(o=ref["o"], lse=ref["lse"])  # the forward the oracle's chain rule ran on
    model = rounded_backward_grouped(f, fwd, ref["gate"], ratio, causal=causal, scale=scale)
    return ref, model


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


@pytest.mark.parametrize("B,N,h,ratio,hkv", [(1, 200, 6, 3, 2), (1, 300, 8, 4, 1), (2, 64, 6, 3, 1),
                                              (1, 1, 3, 3, 1), (1, 500, 12, 3, 2), (2, 129, 16, 4, 2),
                                              (2, 7, 6, 3, 2), (1, 260, 4, 2, 1)])
def test_grouped_bwd_parity_small(B, N, h, ratio, hkv):
    """3:1, 4:1 and 2:1 groups, one or several groups per K/V head, one token,
    ragged tails across several 128-key tiles, two batches."""
    t = _inputs(B, N, h, ratio, hkv, 128, 128, seed=9000 + N + h)
    ref, model = _reference(t, ratio)
    _compare(_run_exact_saves(t, ratio, ref), ref, model, bar="bwd")
    _compare(_run(t, ratio), ref, model, bar="step")


@pytest.mark.parametrize("B,N,h,ratio,hkv", [(1, 200, 6, 3, 2), (2, 129, 8, 4, 1), (1, 1, 3, 3, 1)])
def test_grouped_bwd_parity_head_dim_64(B, N, h, ratio, hkv):
    t = _inputs(B, N, h, ratio, hkv, 64, 128, seed=9100 + N + h)
    ref, model = _reference(t, ratio)
    _compare(_run_exact_saves(t, ratio, ref), ref, model, bar="bwd")
    _compare(_run(t, ratio), ref, model, bar="step")


@pytest.mark.parametrize("B,N,h,ratio,hkv,d", [(1, 200, 6, 3, 2, 128), (2, 129, 8, 4, 1, 64),
                                                (1, 300, 6, 3, 1, 128)])
def test_grouped_bwd_parity_not_causal(B, N, h, ratio, hkv, d):
    t = _inputs(B, N, h, ratio, hkv, d, 128, seed=9200 + N + h)
    ref, model = _reference(t, ratio, causal=False)
    _compare(_run_exact_saves(t, ratio, ref, causal=False), ref, model, bar="bwd")
    _compare(_run(t, ratio, causal=False), ref, model, bar="step")


def test_grouped_bwd_ratio_one_is_v2_bwd():
    """Ratio 1 runs the V2 backward: dK, dV and the gate gradients equal
    diffattn_v2_bwd's bit for bit, dQ (fp32 reduce-adds) to rounding."""
    t = synth.v2_inputs(1, 300, 4, 2, 128, 128, seed=9300, device="cuda", with_dout=True)
    _, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True)
    a = bd.diffattn_v2_bwd(t["q"], t["k"], t["v"], t["dout"], sv, x=t["x"], w_lambda=t["w_lambda"], want_dz=True)
    b = bd.diffattn_grouped_bwd(t["q"], t["k"], t["v"], t["dout"], sv, 1, x=t["x"], w_lambda=t["w_lambda"],
                                want_dz=True)
    torch.cuda.synchronize()
    for n in ("dk", "dv", "dz", "dx", "dw"):
        assert torch.equal(a[n], b[n]), n
    assert torch.allclose(a["dq"].float(), b["dq"].float(), rtol=1e-2, atol=1e-3 * float(a["dq"].float().abs().max()))


def test_grouped_bwd_deterministic_parts_repeat():
    """dK, dV (one CTA each) and the gate gradients (fixed-order reductions)
    are bitwise equal on a rerun."""
    t = _inputs(1, 400, 6, 3, 1, 128, 128, seed=9301)
    g1 = _run(t, 3)
    g2 = _run(t, 3)
    for n in ("dk", "dv", "dz", "dx", "dw"):
        assert torch.equal(g1[n], g2[n]), n


def test_grouped_bwd_full_size_b2_n8192_3to1_one_group():
    """B2 N8192, 64 query heads as 16 groups of 3 signal + 1 noise over 8 K/V
    heads, d 128, gate from X [2, 8192, 4096] (the grouped workload) through
    the library; the oracle recomputes one (batch, K/V group) completely: its
    8 query heads' dQ (two signal/noise groups), the group's dK and dV, and dz
    of its 6 output heads."""
    ratio = 3
    t = _inputs(2, 8192, 48, ratio, 8, 128, 4096, seed=1007)
    g = _run(t, ratio)
    b, grp = 0, 6
    qs, ps = slice(8 * grp, 8 * grp + 8), slice(6 * grp, 6 * grp + 6)
    ts = dict(q=t["q"][b:b + 1, :, qs], k=t["k"][b:b + 1, :, grp:grp + 1], v=t["v"][b:b + 1, :, grp:grp + 1],
              x=t["x"][b:b + 1], w_lambda=t["w_lambda"][:, ps], dout=t["dout"][b:b + 1, :, ps])
    ref, model = _reference(ts, ratio)
    sl = dict(dq=(slice(b, b + 1), slice(None), qs), dk=(slice(b, b + 1), slice(None), slice(grp, grp + 1)),
              dv=(slice(b, b + 1), slice(None), slice(grp, grp + 1)), dz=(slice(b, b + 1), slice(None), ps))
    _compare(g, ref, model, names=ATTN + ("dz",), bar="step", sl=sl)
