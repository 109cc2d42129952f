"""GPU parity through the C ABI for the V1 decode (split-KV kernel over two K
caches and a shared V cache, then the merge with the difference, RMSNorm and
scale) against the fp64 oracle: ragged lengths, explicit split counts, one
key, exact cancellation, the bounds report, and a large cache on sampled
sequences.  Bar: max|diff| <= 2e-2 * RMS(V) (bf16 I/O, fp32 accumulation)."""

import math

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from oracle import diffattn_oracle as orc

pytestmark = pytest.mark.gpu
TOL = 2e-2
LAMS = ("lq1", "lk1", "lq2", "lk2")


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _run(t, li, **kw):
    out = bd.diffattn_v1_decode(t["q1"], t["q2"], t["k1_cache"], t["k2_cache"], t["v_cache"],
                                *(t[n] for n in LAMS), li, seqlens=t["seqlens"], **kw)
    torch.cuda.synchronize()
    return out


def _check(t, li, out, batches=None, w=None, scale=None, eps=1e-5):
    B = t["q1"].shape[0]
    batches = range(B) if batches is None else batches
    sl = [int(x) for x in t["seqlens"].cpu()]
    o = f64(out)
    worst = 0.0
    for b in batches:
        L = sl[b]
        ref = orc.v1_decode(f64(t["q1"][b:b + 1]), f64(t["q2"][b:b + 1]), f64(t["k1_cache"][b:b + 1, :L]),
                            f64(t["k2_cache"][b:b + 1, :L]), f64(t["v_cache"][b:b + 1, :L]), [L],
                            *(f64(t[n]) for n in LAMS), float(np.float32(li)),
                            rms_weight=None if w is None else f64(w), scale=scale, eps=eps)
        for h in range(t["q1"].shape[1]):
            v = f64(t["v_cache"][b, :L, h])
            tol = TOL * float(np.sqrt(np.mean(v * v)))
            worst = max(worst, float(np.max(np.abs(o[b, h] - ref["y"][0, h]))) / tol)
    assert worst <= 1.0, worst


@pytest.mark.parametrize("B,L,H,seqlens,splits,layer", [
    (2, 200, 2, [200, 77], 0, 1),
    (3, 1000, 4, [1000, 513, 64], 3, 5),
    (1, 1, 1, [1], 0, 28),
    (2, 4096, 2, [4096, 4000], 7, 14),
    (1, 2500, 3, [2500], 1, 2),
])
def test_v1_decode_parity(B, L, H, seqlens, splits, layer):
    t = synth.v1_decode_inputs(B, L, H, 128, 256, seed=6000 + L + H, device="cuda", seqlens=seqlens)
    li = bd.diffattn_lambda_init(layer)
    _check(t, li, _run(t, li, num_splits=splits))


@pytest.mark.parametrize("B,L,H,seqlens,splits,layer", [
    (2, 200, 2, [200, 77], 0, 1),
    (3, 1000, 4, [1000, 513, 1], 3, 5),
])
def test_v1_decode_parity_head_dims_64_128(B, L, H, seqlens, splits, layer):
    t = synth.v1_decode_inputs(B, L, H, 64, 128, seed=6100 + L + H, device="cuda", seqlens=seqlens)
    li = bd.diffattn_lambda_init(layer)
    _check(t, li, _run(t, li, num_splits=splits))


def test_v1_decode_parity_rms_weight():
    t = synth.v1_decode_inputs(2, 700, 3, 128, 256, seed=6200, device="cuda", seqlens=[700, 333])
    w = 0.5 + torch.rand(256, generator=torch.Generator().manual_seed(6201), dtype=torch.float32).cuda()
    li = bd.diffattn_lambda_init(4)
    _check(t, li, _run(t, li, num_splits=3, rms_weight=w), w=w)


def test_v1_decode_split_count_invariance():
    """The split-KV partition changes only rounding: 1 split vs many agree."""
    t = synth.v1_decode_inputs(2, 3000, 2, 128, 256, seed=61, device="cuda")
    li = bd.diffattn_lambda_init(3)
    a = _run(t, li, num_splits=1).float()
    b = _run(t, li, num_splits=11).float()
    assert float((a - b).abs().max()) <= 2e-2 * float(a.pow(2).mean().sqrt())


def test_v1_decode_exact_cancellation():
    """q1 = q2, K1 = K2 and lambda = exp(ln 2) - exp(0) + 0 = 1: both streams
    run identical arithmetic, so O and Y are exactly zero."""
    t = synth.v1_decode_inputs(2, 700, 2, 128, 256, seed=62, device="cuda")
    lq1 = torch.zeros(128, device="cuda")
    lq1[0] = 1.0
    lk1 = torch.zeros(128, device="cuda")
    lk1[0] = math.log(2.0)
    z = torch.zeros(128, device="cuda")
    out = bd.diffattn_v1_decode(t["q1"], t["q1"], t["k1_cache"], t["k1_cache"], t["v_cache"], lq1, lk1, z, z,
                                0.0, num_splits=3)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_v1_decode_bad_seqlen_reports_bounds():
    t = synth.v1_decode_inputs(2, 128, 2, 128, 256, seed=63, device="cuda", seqlens=[128, 129])
    out = bd.diffattn_v1_decode(t["q1"], t["q2"], t["k1_cache"], t["k2_cache"], t["v_cache"],
                                *(t[n] for n in LAMS), 0.2, seqlens=t["seqlens"])
    assert bd.diffattn_get_device_status() == bd.DA_ERR_BOUNDS
    assert torch.count_nonzero(out[1]).item() == 0
    assert bd.diffattn_get_device_status() == bd.DA_OK


def test_v1_decode_large_cache_sampled():
    """B64, cache 32768, 16 heads, d_qk 128, d_v 256 (the V1 decode workload,
    default split count); the oracle on three whole sequences."""
    t = synth.v1_decode_inputs(64, 32768, 16, 128, 256, seed=1006, device="cuda")
    li = bd.diffattn_lambda_init(1)
    out = _run(t, li)
    _check(t, li, out, batches=[0, 29, 63])
    del t
    torch.cuda.empty_cache()
