"""GPU parity through the C ABI for grouped differential attention (the V2
attention kernel over all query heads, then the group combination) against
the fp64 oracle: 3:1 and 4:1 groups, several groups per K/V head, ragged
tails, one token, ratio 1 against the V2 forward, exact cancellation, and the
full-size workload on sampled rows.  Bar: max|diff| <= 2e-2 * RMS(V)."""

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from oracle import diffattn_oracle as orc
from bf16_model import rounded_grouped_forward
from ratio_log import record
from sampling import tile_rows

pytestmark = pytest.mark.gpu
TOL = 2e-2


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _check(t, ratio, out, rows=None, batches=None, groups=None, causal=True, scale=None):
    """out within 2e-2 * RMS(V) per element.  A row beyond that is held to 3
    times the grouped rounding model's own error on that row instead
    (bf16_model.rounded_grouped_forward: bf16 P, the per-head outputs stored
    in bf16 for the combine, the output rounded).  Those three storage points
    in series can reach the bar at elements of 2-3 RMS(V) under a sharp
    softmax.  The model runs only for groups that need it, and the ratio log
    counts such rows."""
    B, N, Hq, d = t["q"].shape
    hkv = t["k"].shape[2]
    G = Hq // hkv
    batches = range(B) if batches is None else batches
    groups = range(Hq // (ratio + 1)) if groups is None else groups
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    o = f64(out)
    worst = 0.0
    model_rows = 0
    for b in batches:
        for g in groups:
            c = g * (ratio + 1) // G
            qs = slice(g * (ratio + 1), (g + 1) * (ratio + 1))
            ps = slice(g * ratio, (g + 1) * ratio)
            ref = orc.grouped_forward(f64(t["q"][b:b + 1, :, qs]), f64(t["k"][b:b + 1, :, c:c + 1]),
                                      f64(t["v"][b:b + 1, :, c:c + 1]), gate[b:b + 1, :, ps], ratio, rows=rows,
                                      causal=causal, scale=scale)
            r = ref["rows"]
            tol = TOL * float(np.sqrt(np.mean(f64(t["v"][b, :, c]) ** 2)))
            err = np.max(np.abs(o[b, r, ps] - ref["out"][0]), axis=(1, 2))
            allowed = np.full_like(err, tol)
            if np.max(err) > tol:
                exact = orc.grouped_forward(f64(t["q"][b:b + 1, :, qs]), f64(t["k"][b:b + 1, :, c:c + 1]),
                                            f64(t["v"][b:b + 1, :, c:c + 1]), gate[b:b + 1, :, ps], ratio,
                                            causal=causal, scale=scale)["out"][0]
                model = rounded_grouped_forward(f64(t["q"][b, :, qs]), f64(t["k"][b, :, c]), f64(t["v"][b, :, c]),
                                                gate[b, :, ps], ratio, scale=scale, causal=causal)
                merr = np.max(np.abs(model[r] - exact[r]), axis=(1, 2))
                allowed = np.maximum(tol, 3 * merr)
                model_rows += int(np.sum(allowed > tol))
            worst = max(worst, float(np.max(err / allowed)))
    record({"out": worst, "rows_on_model_bar": model_rows})
    assert worst <= 1.0, worst


@pytest.mark.parametrize("B,N,h,ratio,hkv", [(1, 200, 6, 3, 2), (1, 300, 8, 4, 1), (2, 64, 6, 3, 1),
                                              (1, 1, 3, 3, 1), (1, 500, 12, 3, 2), (2, 129, 16, 4, 2),
                                              (2, 7, 6, 3, 2)])
def test_grouped_parity_small(B, N, h, ratio, hkv):
    t = synth.grouped_inputs(B, N, h, ratio, hkv, 128, 128, seed=8000 + N + h, device="cuda")
    out = bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], ratio, x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    _check(t, ratio, out)


@pytest.mark.parametrize("B,N,h,ratio,hkv", [(1, 200, 6, 3, 2), (2, 129, 8, 4, 1)])
def test_grouped_parity_head_dim_64(B, N, h, ratio, hkv):
    t = synth.grouped_inputs(B, N, h, ratio, hkv, 64, 128, seed=8100 + N + h, device="cuda")
    out = bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], ratio, x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    _check(t, ratio, out)


@pytest.mark.parametrize("B,N,h,ratio,hkv,d", [(1, 200, 6, 3, 2, 128), (2, 129, 8, 4, 1, 64)])
def test_grouped_parity_not_causal(B, N, h, ratio, hkv, d):
    t = synth.grouped_inputs(B, N, h, ratio, hkv, d, 128, seed=8200 + N + h, device="cuda")
    out = bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], ratio, x=t["x"], w_lambda=t["w_lambda"], causal=False)
    torch.cuda.synchronize()
    _check(t, ratio, out, causal=False)


def test_grouped_ratio_one_matches_v2():
    """ratio 1 is the V2 forward (which combines in fp32 rather than from
    bf16 head outputs: equal up to that rounding, well inside the bar)."""
    t = synth.v2_inputs(1, 300, 4, 2, 128, 128, seed=81, device="cuda")
    a = bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], 1, x=t["x"], w_lambda=t["w_lambda"]).float()
    b = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"]).float()
    torch.cuda.synchronize()
    assert float((a - b).abs().max()) <= TOL * float(t["v"].float().pow(2).mean().sqrt())


def test_grouped_exact_cancellation():
    """Every signal query equal to its group's noise query and gate 1: zero."""
    ratio = 3
    t = synth.grouped_inputs(1, 333, 6, ratio, 2, 128, 128, seed=82, device="cuda")
    q = t["q"].clone()
    for g in range(2):
        for i in range(ratio):
            q[:, :, g * (ratio + 1) + i] = q[:, :, g * (ratio + 1) + ratio]
    gate = torch.ones((1, 333, 6), dtype=torch.float32, device="cuda")
    out = bd.diffattn_grouped_fwd(q, t["k"], t["v"], ratio, gate=gate)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_grouped_saves_heads_and_lse():
    """The per-head outputs and LSEs the call can save match the oracle."""
    ratio = 4
    t = synth.grouped_inputs(1, 260, 8, ratio, 1, 128, 128, seed=83, device="cuda")
    Hq = 10
    heads = torch.empty((1, 260, Hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, Hq, 260), dtype=torch.float32, device="cuda")
    bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], ratio, x=t["x"], w_lambda=t["w_lambda"], o_heads=heads,
                            lse=lse)
    torch.cuda.synchronize()
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    ref = orc.grouped_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), gate, ratio)
    tol = TOL * float(np.sqrt(np.mean(f64(t["v"]) ** 2)))
    assert float(np.max(np.abs(f64(heads) - ref["o"]))) <= tol
    assert float(np.max(np.abs(f64(lse) - ref["lse"]))) <= 1e-3


def test_grouped_full_size_sampled():
    """B2 N8192, 64 query heads as 16 groups of 3 signal + 1 noise over 8 K/V
    heads, d 128, gate from X [2, 8192, 4096]: every batch and group, the
    first, last and one seeded interior row of every 128-row query tile."""
    ratio = 3
    t = synth.grouped_inputs(2, 8192, 48, ratio, 8, 128, 4096, seed=1007, device="cuda")
    out = bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], ratio, x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    _check(t, ratio, out, rows=tile_rows(8192, seed=7))
