"""GPU parity through the C ABI for the V2 forward (tcgen05 kernel) against
the fp64 oracle: small shapes spanning several 128-row tiles and ragged
tails, the edge cases (one token, one pair, gate given or computed), exact
cancellation, and the full-size workload on sampled rows.  Bar: max|diff| <=
2e-2 * RMS(V) (bf16 I/O, fp32 accumulation)."""

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from oracle import diffattn_oracle as orc
from ratio_log import record
from sampling import tile_rows

pytestmark = pytest.mark.gpu
TOL = 2e-2


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rms(a):
    return float(np.sqrt(np.mean(np.square(a))))


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _check_pairs(t, out, gate, pairs=None, rows=None, lse=None, causal=True, scale=None):
    B, N, H2, d = t["q"].shape
    hkv = t["k"].shape[2]
    G = H2 // hkv
    pairs = range(H2 // 2) if pairs is None else pairs
    o = f64(out)
    worst = 0.0
    for b in range(B):
        for p in pairs:
            g = (2 * p) // G
            ref = orc.v2_forward(f64(t["q"][b:b + 1, :, 2 * p:2 * p + 2]), f64(t["k"][b:b + 1, :, g:g + 1]),
                                 f64(t["v"][b:b + 1, :, g:g + 1]), gate[b:b + 1, :, p:p + 1], rows=rows,
                                 causal=causal, scale=scale)
            got = o[b, ref["rows"], p]
            tol = TOL * rms(f64(t["v"][b, :, g]))
            worst = max(worst, float(np.max(np.abs(got - ref["out"][0, :, 0]))) / tol)
            if lse is not None:
                lg = f64(lse[b, 2 * p:2 * p + 2][:, ref["rows"]])
                assert np.max(np.abs(lg - ref["lse"][0])) <= 1e-3
    record({"out": worst})
    assert worst <= 1.0, worst


@pytest.mark.parametrize("B,N,h,hkv", [(1, 200, 4, 2), (2, 384, 2, 1), (1, 129, 4, 4), (1, 1, 2, 1),
                                        (2, 1000, 8, 2), (1, 640, 16, 2), (2, 7, 2, 1), (1, 64, 4, 2)])
def test_v2_fwd_parity_small(B, N, h, hkv):
    t = synth.v2_inputs(B, N, h, hkv, 128, 128, seed=3000 + N + h, device="cuda")
    lse = torch.empty((B, 2 * h, N), dtype=torch.float32, device="cuda")
    out = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], lse=lse)
    torch.cuda.synchronize()
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    _check_pairs(t, out, gate, lse=lse)


@pytest.mark.parametrize("B,N,h,hkv", [(1, 200, 4, 2), (2, 300, 2, 1), (1, 1, 2, 1), (1, 700, 8, 2)])
def test_v2_fwd_parity_head_dim_64(B, N, h, hkv):
    """Head dim 64 (one 64-column box per tile row, PV with N = 64): ragged
    tails, one token, several query tiles; LSE and per-head saves checked."""
    t = synth.v2_inputs(B, N, h, hkv, 64, 128, seed=3100 + N + h, device="cuda")
    out, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True)
    torch.cuda.synchronize()
    lse, heads = sv["lse"], sv["o_heads"]
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    _check_pairs(t, out, gate, lse=lse)
    # each head's normalised output: the pair with gate 0 is that head alone
    G = 2 * h // hkv
    for j in (0, 2 * h - 1):
        g = j // G
        ref = orc.v2_forward(f64(t["q"][:1, :, [j, j]]), f64(t["k"][:1, :, g:g + 1]), f64(t["v"][:1, :, g:g + 1]),
                             np.zeros((1, N, 1)))
        tol = TOL * rms(f64(t["v"][0, :, g]))
        assert np.max(np.abs(f64(heads[0, :, j]) - ref["out"][0, :, 0])) <= tol


def test_v2_fwd_exact_cancellation_head_dim_64():
    """Head dim 64: equal even and odd queries with gate 1 give exactly zero."""
    t = synth.v2_inputs(1, 333, 4, 2, 64, 128, seed=34, device="cuda")
    q = t["q"].clone()
    q[:, :, 1::2] = q[:, :, 0::2]
    gate = torch.ones((1, 333, 4), dtype=torch.float32, device="cuda")
    out = bd.diffattn_v2_fwd(q, t["k"], t["v"], gate=gate)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


@pytest.mark.parametrize("B,N,h,hkv,d", [(1, 200, 4, 2, 128), (2, 129, 2, 1, 64), (1, 1, 2, 1, 128),
                                          (1, 384, 4, 4, 128), (1, 700, 8, 2, 64)])
def test_v2_fwd_parity_not_causal(B, N, h, hkv, d):
    """Every query attends every key: all key tiles per item, the ragged last
    key tile masked at N."""
    t = synth.v2_inputs(B, N, h, hkv, d, 128, seed=3200 + N + h, device="cuda")
    out, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True,
                                 causal=False)
    torch.cuda.synchronize()
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    _check_pairs(t, out, gate, lse=sv["lse"], causal=False)


@pytest.mark.parametrize("causal", [True, False])
def test_v2_fwd_late_large_scores_rescale(causal):
    """Keys from 256 on scaled by 30: their scores exceed the first tile's
    running max by far more than the softmax's stale-max guard allows, so the
    rows re-normalise mid-sequence (new max, O and l rescaled)."""
    t = synth.v2_inputs(1, 500, 2, 1, 128, 128, seed=3300, device="cuda")
    t["k"][:, 256:] *= 30.0
    out, sv = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], save=True,
                                 causal=causal)
    torch.cuda.synchronize()
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    _check_pairs(t, out, gate, lse=sv["lse"], causal=causal)


def test_v2_fwd_gate_given_equals_x_path():
    t = synth.v2_inputs(1, 300, 4, 2, 128, 256, seed=31, device="cuda")
    gate = bd.diffattn_v2_gate(t["x"], t["w_lambda"])
    o1 = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], gate=gate)
    o2 = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_v2_fwd_exact_cancellation():
    """Odd query = even query and gate 1: bit-exact zero (both heads run the
    same MMAs and softmax arithmetic)."""
    t = synth.v2_inputs(1, 333, 4, 2, 128, 128, seed=32, device="cuda")
    q = t["q"].clone()
    q[:, :, 1::2] = q[:, :, 0::2]
    gate = torch.ones((1, 333, 4), dtype=torch.float32, device="cuda")
    out = bd.diffattn_v2_fwd(q, t["k"], t["v"], gate=gate)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_v2_fwd_gate_zero_is_even_head_attention():
    """gate = 0: the output is plain causal attention of the even heads."""
    t = synth.v2_inputs(1, 257, 4, 2, 128, 128, seed=33, device="cuda")
    gate = torch.zeros((1, 257, 4), dtype=torch.float32, device="cuda")
    out = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], gate=gate)
    torch.cuda.synchronize()
    _check_pairs(t, out, np.zeros((1, 257, 4)))


def test_v2_fwd_strided_views():
    """q, k, v as views into one packed [B, N, 2h + 2 h_kv, d] buffer."""
    B, N, h, hkv = 1, 300, 4, 2
    g = torch.Generator(device="cuda").manual_seed(34)
    buf = torch.randn((B, N, 2 * h + 2 * hkv, 128), generator=g, device="cuda").to(torch.bfloat16)
    t = {"q": buf[:, :, :2 * h], "k": buf[:, :, 2 * h:2 * h + hkv], "v": buf[:, :, 2 * h + hkv:]}
    gate = torch.rand((B, N, h), generator=g, device="cuda")
    out = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], gate=gate)
    torch.cuda.synchronize()
    _check_pairs(t, out, f64(gate))


def test_v2_fwd_full_size_sampled():
    """B2, N 8192, 64 query heads / 8 KV heads, d 128, gate from X [2,8192,4096]
    (the prefill workload at full size) against the oracle: every batch and
    pair, the first, last and one seeded interior row of every 128-row query
    tile (every work item of the persistent schedule)."""
    t = synth.v2_inputs(2, 8192, 32, 8, 128, 4096, seed=1003, device="cuda")
    out = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"])
    torch.cuda.synchronize()
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    _check_pairs(t, out, gate, rows=tile_rows(8192, seed=3))
