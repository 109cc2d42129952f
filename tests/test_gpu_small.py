"""GPU parity through the C ABI for the gate, the fp32 V1 path and the V2
decode: CUDA output vs the fp64 oracle, element by element, on seeded
inputs that span several tiles and a ragged tail.

Bars: bf16 I/O with fp32 accumulation: max|diff| <= 2e-2 * RMS(V); the fp32
V1 path: max|diff| <= 1e-4 * RMS(V); the gate (a probability, fp32 output
from exact bf16 products): max|diff| <= 1e-4.
"""

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from oracle import diffattn_oracle as orc
from ratio_log import record

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2
F32_TOL = 1e-4


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rms(a):
    return float(np.sqrt(np.mean(np.square(a))))


def maxdiff(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


# ------------------------------------------------------------------ gate ----

@pytest.mark.parametrize("T,dm,h", [(300, 256, 32), (64, 4096, 32), (1, 64, 8), (129, 128, 64),
                                    (2433, 256, 8), (5000, 512, 48), (16384, 4096, 32), (7001, 128, 64)])
def test_gate_parity(T, dm, h):
    """Few tokens run the cluster-split kernel; 16 or more per SM (with h a
    multiple of 8) the row-range TMA kernel: ragged per-CTA ranges, h = 8 to
    64, d_model from 128 to 4096 (the prefill workload's X [16384, 4096])."""
    g = torch.Generator(device="cuda").manual_seed(100 + T)
    x = torch.randn((T, dm), generator=g, device="cuda").to(torch.bfloat16)
    w = (0.02 * torch.randn((dm, h), generator=g, device="cuda")).to(torch.bfloat16)
    gate = bd.diffattn_v2_gate(x, w)
    torch.cuda.synchronize()
    ref = orc.v2_gate(f64(x), f64(w))
    assert maxdiff(f64(gate), ref) <= 1e-4


def test_gate_strided_rows_many_tokens():
    """X as a strided view (row stride 4096 + 64 elements) on the row-range
    kernel: the gate of the view equals the gate of a contiguous copy."""
    g = torch.Generator(device="cuda").manual_seed(7)
    buf = torch.randn((4000, 4160), generator=g, device="cuda").to(torch.bfloat16)
    x = buf[:, :4096]
    w = (0.02 * torch.randn((4096, 32), generator=g, device="cuda")).to(torch.bfloat16)
    a = bd.diffattn_v2_gate(x, w)
    b = bd.diffattn_v2_gate(x.contiguous(), w)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert maxdiff(f64(a), orc.v2_gate(f64(x), f64(w))) <= 1e-4


# --------------------------------------------------------------- V1 fp32 ----

@pytest.mark.parametrize("B,N,H,dqk,dv,layer", [(1, 64, 2, 16, 32, 1), (2, 77, 3, 20, 64, 14),
                                                 (1, 1, 1, 16, 32, 2), (1, 130, 2, 128, 256, 28)])
def test_v1_fwd_f32_parity(B, N, H, dqk, dv, layer):
    t = synth.v1_inputs(B, N, H, dqk, dv, dtype="f32", seed=1000 + N, device="cuda")
    li = bd.diffattn_lambda_init(layer)
    out, sv = bd.diffattn_v1_fwd(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], t["lq1"], t["lk1"],
                                 t["lq2"], t["lk2"], li, save=True)
    torch.cuda.synchronize()
    ref = orc.v1_forward(*(f64(t[n]) for n in ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2",
                                                "lk2")), float(np.float32(li)))
    tol = F32_TOL * rms(f64(t["v"]))
    assert maxdiff(f64(out), ref["y"]) <= tol
    assert maxdiff(f64(sv["o2"]), ref["o2"]) <= tol
    assert maxdiff(f64(sv["lse1"]), ref["lse1"]) <= 1e-4
    assert maxdiff(f64(sv["lse2"]), ref["lse2"]) <= 1e-4
    assert np.max(np.abs(f64(sv["rstd"]) / ref["rstd"] - 1)) <= 1e-4
    assert abs(float(sv["lam"][0]) - ref["lam"]) <= 1e-6


def test_v1_fwd_f32_rms_weight():
    t = synth.v1_inputs(2, 77, 3, 20, 64, dtype="f32", seed=1077, device="cuda")
    w = 0.5 + torch.rand(64, generator=torch.Generator().manual_seed(1078), dtype=torch.float32).cuda()
    li = bd.diffattn_lambda_init(3)
    out = bd.diffattn_v1_fwd(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], t["lq1"], t["lk1"],
                             t["lq2"], t["lk2"], li, rms_weight=w)
    torch.cuda.synchronize()
    ref = orc.v1_forward(*(f64(t[n]) for n in ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2",
                                                "lk2")), float(np.float32(li)), rms_weight=f64(w))
    assert maxdiff(f64(out), ref["y"]) <= F32_TOL * rms(f64(t["v"]))


def test_v1_fwd_f32_not_causal():
    """The fp32 SIMT path without the causal mask: every query sees every key."""
    t = synth.v1_inputs(2, 77, 3, 20, 64, dtype="f32", seed=1177, device="cuda")
    li = bd.diffattn_lambda_init(5)
    out, sv = bd.diffattn_v1_fwd(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], t["lq1"], t["lk1"],
                                 t["lq2"], t["lk2"], li, save=True, causal=False)
    torch.cuda.synchronize()
    ref = orc.v1_forward(*(f64(t[n]) for n in ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2",
                                                "lk2")), float(np.float32(li)), causal=False)
    tol = F32_TOL * rms(f64(t["v"]))
    assert maxdiff(f64(out), ref["y"]) <= tol
    assert maxdiff(f64(sv["o2"]), ref["o2"]) <= tol
    assert maxdiff(f64(sv["lse1"]), ref["lse1"]) <= 1e-4


def test_v1_fwd_f32_exact_cancellation():
    """Q1 = Q2, K1 = K2 and lambda = 1: both streams run the same arithmetic,
    so the difference and the output are exactly zero."""
    t = synth.v1_inputs(1, 64, 2, 16, 32, dtype="f32", seed=7, device="cuda")
    z = torch.zeros_like(t["lq1"])
    out = bd.diffattn_v1_fwd(t["q1"], t["q1"], t["k1"], t["k1"], t["v"], z, z, z, z, 1.0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


# ---------------------------------------------------------------- decode ----

def _decode_check(t, out, gate=None, batches=None, scale=None):
    q, kc, vc = f64(t["q"]), t["k_cache"], t["v_cache"]
    sl = t["seqlens"].cpu().numpy()
    if gate is None:
        gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    batches = range(q.shape[0]) if batches is None else batches
    o = f64(out)
    worst = 0.0
    for b in batches:
        L = int(sl[b])
        ref = orc.v2_decode(q[b:b + 1], f64(kc[b:b + 1, :L]), f64(vc[b:b + 1, :L]), [L],
                            gate[b:b + 1], scale=scale)
        tol = BF16_TOL * rms(f64(vc[b, :L]))
        d = maxdiff(o[b], ref["out"][0])
        worst = max(worst, d / tol)
    record({"out": worst})
    assert worst <= 1.0, worst


@pytest.mark.parametrize("B,L,h,hkv,seqlens,splits", [
    (3, 1000, 32, 8, [1000, 1, 517], 0),
    (2, 300, 16, 2, [300, 65], 3),      # 16 query heads per group
    (2, 129, 8, 8, [129, 128], 1),      # 2 query heads per group (one pair)
    (1, 4096, 32, 8, [4096], 7),
])
def test_decode_parity(B, L, h, hkv, seqlens, splits):
    t = synth.decode_inputs(B, L, h, hkv, 128, 256, seed=2000 + L, device="cuda", seqlens=seqlens)
    out = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], seqlens=t["seqlens"],
                                x=t["x"], w_lambda=t["w_lambda"], num_splits=splits)
    torch.cuda.synchronize()
    _decode_check(t, out)


@pytest.mark.parametrize("B,L,h,hkv,seqlens,splits", [
    (3, 1000, 32, 8, [1000, 1, 517], 0),
    (2, 300, 16, 2, [300, 65], 3),
    (2, 129, 8, 8, [129, 128], 1),
])
def test_decode_parity_head_dim_64(B, L, h, hkv, seqlens, splits):
    """Head dim 64: key rows of 8 16-byte chunks, 4 feature tiles per warp MMA."""
    t = synth.decode_inputs(B, L, h, hkv, 64, 256, seed=2100 + L, device="cuda", seqlens=seqlens)
    out = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], seqlens=t["seqlens"],
                                x=t["x"], w_lambda=t["w_lambda"], num_splits=splits)
    torch.cuda.synchronize()
    _decode_check(t, out)


def test_decode_gate_given_matches_x_path():
    t = synth.decode_inputs(2, 777, 32, 8, 128, 256, seed=5, device="cuda")
    gate = bd.diffattn_v2_gate(t["x"], t["w_lambda"])
    o1 = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], gate=gate)
    o2 = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_decode_pair_cancellation_exact():
    """Even and odd queries equal and gate = 1: exactly zero output."""
    t = synth.decode_inputs(2, 333, 32, 8, 128, 256, seed=6, device="cuda")
    q = t["q"].clone()
    q[:, 1::2] = q[:, 0::2]
    gate = torch.ones((2, 32), dtype=torch.float32, device="cuda")
    out = bd.diffattn_v2_decode(q, t["k_cache"], t["v_cache"], gate=gate, num_splits=3)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_decode_bad_seqlen_reports_bounds():
    t = synth.decode_inputs(2, 128, 32, 8, 128, 256, seed=8, device="cuda", seqlens=[128, 0])
    out = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], seqlens=t["seqlens"],
                                x=t["x"], w_lambda=t["w_lambda"])
    st = bd.diffattn_get_device_status()
    assert st == bd.DA_ERR_BOUNDS
    assert torch.count_nonzero(out[1]).item() == 0
    assert bd.diffattn_get_device_status() == bd.DA_OK  # cleared by the read


def test_decode_full_size_sampled():
    """B64, cache 32768, 8 KV heads, 64 query heads, d 128 (the decode
    workload at full size, default split count); the oracle on 17 of the 64
    sequences, every fourth plus the last, all 64 query heads each."""
    t = synth.decode_inputs(64, 32768, 32, 8, 128, 4096, seed=1004, device="cuda")
    out = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], x=t["x"],
                                w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    _decode_check(t, out, gate=gate, batches=list(range(0, 64, 4)) + [63])
    del t
    torch.cuda.empty_cache()
