"""Pins for the fp64 oracle: each test checks it against something other than
itself (a closed form, a library routine in a special case, an exact
invariant, brute force, finite differences), chosen so that a dropped term, a
wrong sign, a swapped stream or head, or a wrong scale fails at least one.

Sources: "Differential Transformer | ICLR 2025 Oral" (dainus.ai) and
"Differential Transformer V2" (pogovet.com); sections named per test.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.linalg import hadamard

from oracle import diffattn_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_printed_values.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _sdpa(q, k, v, causal=True):
    """Library softmax attention (torch SDPA, float64, CPU) of one head:
    q [N,d], k [N,d], v [N,dv]."""
    qt = torch.from_numpy(np.ascontiguousarray(q))[None, None]
    kt = torch.from_numpy(np.ascontiguousarray(k))[None, None]
    vt = torch.from_numpy(np.ascontiguousarray(v))[None, None]
    return F.scaled_dot_product_attention(qt, kt, vt, is_causal=causal)[0, 0].numpy()


def _v1_rand(B=2, N=9, H=3, dqk=4, dv=8, seed=0, lam_std=0.1):
    r = _rng(seed)
    t = {n: r.standard_normal((B, N, H, dqk)) for n in ("q1", "q2", "k1", "k2")}
    t["v"] = r.standard_normal((B, N, H, dv))
    for n in ("lq1", "lk1", "lq2", "lk2"):
        t[n] = lam_std * r.standard_normal(dqk)
    return t


def _v1(t, lam_init, **kw):
    return orc.v1_forward(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], t["lq1"],
                          t["lk1"], t["lq2"], t["lk2"], lam_init, **kw)


# ---------------------------------------------------------------- lambda ----

def test_lambda_init_closed_form():
    """[P1] 'λ의 역할과 학습': 0.8 - 0.6 exp(-0.3 (l-1)); l = 1 is the first layer."""
    g = json.load(open(GOLDEN))["lambda_init"]
    assert g["first_layer"] == 1
    assert orc.lambda_init(1) == pytest.approx(0.2, abs=1e-15)       # e^0 = 1
    assert orc.lambda_init(2) == pytest.approx(0.8 - 0.6 / math.e ** 0.3, abs=1e-15)
    # the schedule rises monotonically toward 0.8 with depth
    vals = [orc.lambda_init(l) for l in range(1, 29)]
    assert all(b > a for a, b in zip(vals, vals[1:]))
    assert 0.7998 < vals[-1] < 0.8
    # ln-space check: 0.8 - lambda_init(l) = 0.6 e^{-0.3 (l-1)}
    for l in (3, 5, 10, 14, 20, 28):
        assert math.log((0.8 - orc.lambda_init(l)) / 0.6) == pytest.approx(-0.3 * (l - 1), abs=1e-12)


def test_lambda_full_closed_forms():
    """Reparameterisation exp(lq1.lk1) - exp(lq2.lk2) + lambda_init."""
    z = np.zeros(5)
    assert orc.lambda_full(z, z, z, z, 0.37) == pytest.approx(0.37, abs=1e-15)
    e0 = np.eye(5)[0]
    # exp(ln 2) - exp(ln 3) + 0.2 = -0.8 ; sign of the second term pinned
    lam = orc.lambda_full(e0, math.log(2.0) * e0, e0, math.log(3.0) * e0, 0.2)
    assert lam == pytest.approx(-0.8, abs=1e-14)
    # orthogonal vectors give a zero dot product
    assert orc.lambda_full(e0, np.eye(5)[1], z, z, 0.5) == pytest.approx(0.5, abs=1e-15)


# --------------------------------------------------------------- softmax ----

def test_softmax_rows_nonnegative_sum_to_one():
    """[P1] 'Softmax 어텐션의 구조적 한계': weights are non-negative and sum to 1."""
    r = _rng(1)
    q, k = r.standard_normal((17, 6)), r.standard_normal((17, 6))
    for causal in (True, False):
        a, lse = orc.attention_maps(q, k, 0.4, causal)
        assert (a >= 0).all()
        np.testing.assert_allclose(a.sum(1), 1.0, atol=1e-14)
        if causal:
            assert np.all(np.triu(a, 1) == 0)
        s = 0.4 * q @ k.T
        if causal:
            s = np.where(np.tril(np.ones_like(s)) > 0, s, -np.inf)
        np.testing.assert_allclose(lse, np.log(np.exp(s).sum(1)), rtol=1e-13)


# ------------------------------------------------------------- V1 forward ---

def test_v1_lambda_zero_is_library_attention():
    """lambda = 0 (zero vectors, lambda_init = 0): the pre-norm output is plain
    softmax attention of stream 1 ([P1] formula), compared with torch SDPA."""
    t = _v1_rand(seed=2)
    for n in ("lq1", "lk1", "lq2", "lk2"):
        t[n] = np.zeros_like(t[n])
    out = _v1(t, 0.0)
    assert out["lam"] == 0.0
    for b in range(2):
        for h in range(3):
            ref = _sdpa(t["q1"][b, :, h], t["k1"][b, :, h], t["v"][b, :, h])
            np.testing.assert_allclose(out["o"][b, :, h], ref, atol=1e-12)
            ref2 = _sdpa(t["q2"][b, :, h], t["k2"][b, :, h], t["v"][b, :, h])
            np.testing.assert_allclose(out["o2"][b, :, h], ref2, atol=1e-12)


def test_v1_lambda_zero_not_causal_is_library_attention():
    """As above without the causal mask: every query sees every key."""
    t = _v1_rand(seed=5)
    for n in ("lq1", "lk1", "lq2", "lk2"):
        t[n] = np.zeros_like(t[n])
    out = _v1(t, 0.0, causal=False)
    for b in range(2):
        for h in range(3):
            ref = _sdpa(t["q1"][b, :, h], t["k1"][b, :, h], t["v"][b, :, h], causal=False)
            np.testing.assert_allclose(out["o"][b, :, h], ref, atol=1e-12)


def test_v1_identical_streams_scale_by_one_minus_lambda():
    """Q2 = Q1, K2 = K1: both maps are equal, so O = (1 - lambda) * attention."""
    t = _v1_rand(seed=3)
    t["q2"], t["k2"] = t["q1"].copy(), t["k1"].copy()
    out = _v1(t, 0.35)
    lam = out["lam"]
    for b in range(2):
        for h in range(3):
            ref = _sdpa(t["q1"][b, :, h], t["k1"][b, :, h], t["v"][b, :, h])
            np.testing.assert_allclose(out["o"][b, :, h], (1 - lam) * ref, atol=1e-12)


def test_v1_uniform_second_map_pins_stream_order():
    """Q2 = 0 makes map 2 the causal mean (closed form: cumulative mean of V), so
    O = attention(Q1, K1, V) - lambda * cummean(V); a swapped stream fails."""
    t = _v1_rand(seed=4)
    t["q2"] = np.zeros_like(t["q2"])
    out = _v1(t, 0.5)
    lam = out["lam"]
    n = np.arange(1, 10)[:, None]
    for b in range(2):
        for h in range(3):
            V = t["v"][b, :, h]
            ref = _sdpa(t["q1"][b, :, h], t["k1"][b, :, h], V) - lam * np.cumsum(V, 0) / n
            np.testing.assert_allclose(out["o"][b, :, h], ref, atol=1e-12)


def test_v1_exact_cancellation():
    """Q1 = Q2, K1 = K2, lambda = 1: O is exactly zero, so Y = 0 (0 / sqrt(eps))."""
    t = _v1_rand(seed=5)
    t["q2"], t["k2"] = t["q1"].copy(), t["k1"].copy()
    for n in ("lq1", "lk1", "lq2", "lk2"):
        t[n] = np.zeros_like(t[n])
    out = _v1(t, 1.0)
    assert out["lam"] == 1.0
    assert np.all(out["o"] == 0.0) and np.all(out["y"] == 0.0)


def test_v1_per_head_rms_and_scale():
    """[P2] §1: per-head RMSNorm, then the (1 - lambda_init) scale.  Every
    (b, n, h) row of Y has RMS c * sqrt(ms / (ms + eps)) with c = 1 - lambda_init,
    i.e. just under c; a norm over the wrong axis or a scale of lambda_init fails."""
    t = _v1_rand(seed=6, dv=16)
    li = orc.lambda_init(3)
    out = _v1(t, li)
    c = 1.0 - li
    rms_y = np.sqrt(np.mean(out["y"] ** 2, axis=-1))
    ms_o = np.mean(out["o"] ** 2, axis=-1)
    assert np.all(rms_y <= c * (1 + 1e-12))
    assert np.all(rms_y >= c * np.sqrt(1 - 1e-5 / ms_o.min()) * (1 - 1e-12))
    # rstd is 1/sqrt(ms + eps) per (b, h, n)
    np.testing.assert_allclose(out["rstd"], 1 / np.sqrt(ms_o.transpose(0, 2, 1) + 1e-5), rtol=1e-12)


def test_v1_rms_weight_scales_features():
    """The RMSNorm weight multiplies each feature of the normalised output:
    Y_w = w * Y_unit exactly (its definition), the pre-norm O and the saves
    unchanged; the decode applies it the same way."""
    t = _v1_rand(seed=9)
    w = _rng(10).uniform(0.5, 1.5, t["v"].shape[-1])
    base, wtd = _v1(t, 0.3), _v1(t, 0.3, rms_weight=w)
    np.testing.assert_allclose(wtd["y"], base["y"] * w, rtol=1e-15, atol=0)
    for n in ("o", "o2", "rstd", "lse1", "lse2"):
        assert np.array_equal(wtd[n], base[n]), n
    B, N, H, dqk = t["q1"].shape
    dec = orc.v1_decode(t["q1"][:, -1], t["q2"][:, -1], t["k1"], t["k2"], t["v"], [N] * B,
                        t["lq1"], t["lk1"], t["lq2"], t["lk2"], 0.3, rms_weight=w)
    np.testing.assert_allclose(dec["y"], wtd["y"][:, -1], rtol=1e-12, atol=1e-14)


def test_v1_first_row_closed_form():
    """Causal row 0 sees only key 0: both maps are [1], O[0] = (1 - lambda) V[0]."""
    t = _v1_rand(seed=7, N=5)
    li = orc.lambda_init(5)
    out = _v1(t, li)
    lam = out["lam"]
    v0 = t["v"][:, 0]
    o0 = (1 - lam) * v0
    y0 = (1 - li) * o0 / np.sqrt(np.mean(o0 ** 2, -1, keepdims=True) + 1e-5)
    np.testing.assert_allclose(out["y"][:, 0], y0, atol=1e-13)


def test_v1_brute_force_scalar_loops():
    """Pure-Python scalar loops (math.exp) on a tiny case vs the matrix oracle."""
    t = _v1_rand(B=1, N=4, H=1, dqk=2, dv=3, seed=8, lam_std=0.5)
    li = 0.3
    out = _v1(t, li)
    Q1, Q2, K1, K2, V = (t[n][0, :, 0] for n in ("q1", "q2", "k1", "k2", "v"))
    lam = (math.exp(sum(a * b for a, b in zip(t["lq1"], t["lk1"])))
           - math.exp(sum(a * b for a, b in zip(t["lq2"], t["lk2"]))) + li)
    s = 1 / math.sqrt(2)
    for i in range(4):
        w = []
        for Q, K in ((Q1, K1), (Q2, K2)):
            sc = [s * sum(Q[i][x] * K[j][x] for x in range(2)) for j in range(i + 1)]
            mx = max(sc)
            ex = [math.exp(v - mx) for v in sc]
            z = sum(ex)
            w.append([e / z for e in ex])
        o = [sum((w[0][j] - lam * w[1][j]) * V[j][c] for j in range(i + 1)) for c in range(3)]
        rr = math.sqrt(sum(x * x for x in o) / 3 + 1e-5)
        y = [(1 - li) * x / rr for x in o]
        np.testing.assert_allclose(out["y"][0, i, 0], y, atol=1e-13)


def test_v1_row_subset_equals_full():
    t = _v1_rand(seed=9, N=12)
    full = _v1(t, 0.2)
    rows = np.array([0, 5, 11])
    sub = _v1(t, 0.2, rows=rows)
    for key in ("y", "o", "o2"):
        np.testing.assert_array_equal(sub[key], full[key][:, rows])
    np.testing.assert_array_equal(sub["lse1"], full["lse1"][:, :, rows])


# ------------------------------------------- context RMS ([P2] §3, §4) ------

def _hadamard_v(n, d):
    """n <= d orthogonal rows with entries +-1 (RMS exactly 1)."""
    return hadamard(d)[:n].astype(np.float64)


def test_plain_attention_rms_bounds_exact():
    """[P2] §3: with uncorrelated unit-RMS values the context RMS lies in
    [1/sqrt(n), 1): uniform map -> 1/sqrt(n), near one-hot -> toward 1.
    Orthogonal (Hadamard) rows make RMS(context) = sqrt(sum_j w_j^2) exact."""
    n, dv = 16, 32
    V = _hadamard_v(n, dv)
    r = _rng(10)
    z = np.zeros((1, n, 1, 4))
    t = dict(q1=z, q2=z, k1=r.standard_normal((1, n, 1, 4)), k2=z,
             v=V[None, :, None, :], lq1=np.zeros(4), lk1=np.zeros(4),
             lq2=np.zeros(4), lk2=np.zeros(4))
    out = _v1(t, 0.0)  # lambda = 0: plain attention
    rms = np.sqrt(np.mean(out["o"][0, :, 0] ** 2, -1))
    np.testing.assert_allclose(rms, 1 / np.sqrt(np.arange(1, n + 1)), rtol=1e-13)
    # random queries: RMS = sqrt(sum w^2), inside [1/sqrt(i+1), 1]
    t["q1"] = 3 * r.standard_normal((1, n, 1, 4))
    out = _v1(t, 0.0)
    a, _ = orc.attention_maps(t["q1"][0, :, 0], t["k1"][0, :, 0], 0.5, True)
    rms = np.sqrt(np.mean(out["o"][0, :, 0] ** 2, -1))
    np.testing.assert_allclose(rms, np.sqrt((a ** 2).sum(1)), rtol=1e-12)
    assert np.all(rms >= 1 / np.sqrt(np.arange(1, n + 1)) - 1e-12)
    assert np.all(rms[1:] < 1.0)
    # a sharp map approaches RMS 1 from below
    kk = 40.0 * np.eye(4)[np.arange(n) % 4]
    t["q1"] = kk[None, :, None, :]
    t["k1"] = kk[None, :, None, :]
    out = _v1(t, 0.0)
    assert np.sqrt(np.mean(out["o"][0, 3, 0] ** 2)) > 0.99


def test_uniform_map_rmsnorm_gain_n8192():
    """[P2] §3 prints about 90.5x for the RMSNorm gain of a uniform map at
    n = 8192 (= sqrt(8192) = 90.51).  Q = 0 gives the uniform map on the last
    causal row; i.i.d. N(0,1) values make RMS = 1/sqrt(n) in expectation
    (chi-square spread over 64 heads x 256 dims: about 0.5 % relative)."""
    g = json.load(open(GOLDEN))["uniform_map_rmsnorm_gain"]
    n = g["seq_len"]
    assert abs(math.sqrt(n) - g["printed_value"]) <= g["printed_precision"]
    r = _rng(11)
    B, H, dqk, dv = 4, 16, 8, 256
    z = np.zeros((B, n, H, dqk))
    v = r.standard_normal((B, n, H, dv))
    t = dict(q1=z, q2=z, k1=z, k2=z, v=v, lq1=np.zeros(dqk), lk1=np.zeros(dqk),
             lq2=np.zeros(dqk), lk2=np.zeros(dqk))
    out = _v1(t, 0.0, rows=np.array([n - 1]), eps=0.0)
    ms = np.mean(out["o"][:, 0] ** 2)
    gain = 1 / math.sqrt(ms)
    assert gain == pytest.approx(g["printed_value"], rel=0.02)
    # with eps = 0 the RMSNorm applies exactly that gain per head: RMS(Y) = 1
    rms_y = np.sqrt(np.mean(out["y"][:, 0] ** 2, axis=-1))
    np.testing.assert_allclose(rms_y, 1.0, rtol=1e-12)


def test_difference_rms_bounds_exact():
    """[P2] §4: the gated difference has context RMS in (0, sqrt 2), exactly
    sqrt(sum_j (a_j - g b_j)^2) for orthogonal unit-RMS value rows."""
    n, d = 16, 32
    r = _rng(12)
    V = _hadamard_v(n, d)
    B, h, hkv = 1, 2, 1
    q = 4 * r.standard_normal((B, n, 2 * h, d))
    k = r.standard_normal((B, n, hkv, d))
    v = V[None, :, None, :]
    gate = r.uniform(0.01, 0.99, (B, n, h))
    out = orc.v2_forward(q, k, v, gate)
    rms = np.sqrt(np.mean(out["out"] ** 2, -1))
    assert np.all(rms > 0) and np.all(rms < math.sqrt(2))
    s = 1 / math.sqrt(d)
    for p in range(h):
        a, _ = orc.attention_maps(q[0, :, 2 * p], k[0, :, 0], s, True)
        b, _ = orc.attention_maps(q[0, :, 2 * p + 1], k[0, :, 0], s, True)
        w = a - gate[0, :, p, None] * b
        np.testing.assert_allclose(rms[0, :, p], np.sqrt((w ** 2).sum(1)), rtol=1e-12)


# ------------------------------------------------------------------ V2 ------

def _v2_rand(B=2, N=11, h=4, hkv=2, d=8, dm=12, seed=20):
    r = _rng(seed)
    return dict(q=r.standard_normal((B, N, 2 * h, d)), k=r.standard_normal((B, N, hkv, d)),
                v=r.standard_normal((B, N, hkv, d)), x=r.standard_normal((B, N, dm)),
                w=0.3 * r.standard_normal((dm, h)))


def test_v2_gate_closed_forms():
    """sigmoid(X W): 0 -> 1/2; X W = ln 3 -> 3/4; X W = -ln 3 -> 1/4."""
    x = np.array([[1.0, 0.0], [0.0, 1.0], [0.0, 0.0]])
    w = np.array([[math.log(3.0), 0.0], [-math.log(3.0), 0.0]])
    g = orc.v2_gate(x, w)
    np.testing.assert_allclose(g, [[0.75, 0.5], [0.25, 0.5], [0.5, 0.5]], atol=1e-15)


def test_v2_gate_zero_is_even_head_library_gqa():
    """gate = 0: Out[p] is the attention of even head 2p on its GQA group's K/V
    (contiguous groups), compared with torch SDPA on repeated K/V heads."""
    t = _v2_rand()
    gate = np.zeros((2, 11, 4))
    out = orc.v2_forward(t["q"], t["k"], t["v"], gate)
    G = 8 // 2
    kr = np.repeat(t["k"], G, axis=2)
    vr = np.repeat(t["v"], G, axis=2)
    for b in range(2):
        for p in range(4):
            ref = _sdpa(t["q"][b, :, 2 * p], kr[b, :, 2 * p], vr[b, :, 2 * p])
            np.testing.assert_allclose(out["out"][b, :, p], ref, atol=1e-12)
            refo = _sdpa(t["q"][b, :, 2 * p + 1], kr[b, :, 2 * p + 1], vr[b, :, 2 * p + 1])
            np.testing.assert_allclose(out["o"][b, :, 2 * p + 1], refo, atol=1e-12)


def test_v2_odd_head_subtracted_with_gate():
    """Even/odd order and gate: with gate g and the odd query replaced by zero
    (uniform causal map), Out = attn(even) - g * cummean(V)."""
    t = _v2_rand(seed=21)
    r = _rng(22)
    gate = r.uniform(0, 1, (2, 11, 4))
    t["q"][:, :, 1::2] = 0.0
    out = orc.v2_forward(t["q"], t["k"], t["v"], gate)
    n = np.arange(1, 12)[:, None]
    for b in range(2):
        for p in range(4):
            gidx = (2 * p) // 4
            ref = (_sdpa(t["q"][b, :, 2 * p], t["k"][b, :, gidx], t["v"][b, :, gidx])
                   - gate[b, :, p, None] * np.cumsum(t["v"][b, :, gidx], 0) / n)
            np.testing.assert_allclose(out["out"][b, :, p], ref, atol=1e-12)


def test_v2_exact_cancellation():
    """Equal even and odd queries with gate 1: the pair output is exactly 0."""
    t = _v2_rand(seed=23)
    t["q"][:, :, 1::2] = t["q"][:, :, 0::2]
    out = orc.v2_forward(t["q"], t["k"], t["v"], np.ones((2, 11, 4)))
    assert np.all(out["out"] == 0.0)


def test_decode_equals_last_causal_row():
    """Decode at position L-1 over a cache of length L is the last row of the
    causal prefill on the same tensors; ragged lengths truncate the cache."""
    t = _v2_rand(seed=24, N=13)
    gate = orc.v2_gate(t["x"], t["w"])
    full = orc.v2_forward(t["q"], t["k"], t["v"], gate)
    seqlens = np.array([13, 6])
    q_dec = np.stack([t["q"][0, 12], t["q"][1, 5]])
    g_dec = np.stack([gate[0, 12], gate[1, 5]])
    dec = orc.v2_decode(q_dec, t["k"], t["v"], seqlens, g_dec)
    np.testing.assert_allclose(dec["out"][0], full["out"][0, 12], atol=1e-12)
    np.testing.assert_allclose(dec["out"][1], full["out"][1, 5], atol=1e-12)
    np.testing.assert_allclose(dec["lse"][0], full["lse"][0, :, 12], atol=1e-12)


def test_v1_decode_equals_last_causal_row():
    """V1 decode at position L-1 is the last row of the causal V1 forward
    (both maps, the difference, the RMSNorm and the scale) on the same
    tensors; ragged lengths truncate both K caches and the V cache."""
    t = _v1_rand(B=2, N=11, H=2, dqk=4, dv=8, seed=25, lam_std=0.4)
    li = 0.45
    full = _v1(t, li)
    seqlens = np.array([11, 4])
    q1 = np.stack([t["q1"][0, 10], t["q1"][1, 3]])
    q2 = np.stack([t["q2"][0, 10], t["q2"][1, 3]])
    dec = orc.v1_decode(q1, q2, t["k1"], t["k2"], t["v"], seqlens, t["lq1"], t["lk1"], t["lq2"],
                        t["lk2"], li)
    np.testing.assert_allclose(dec["y"][0], full["y"][0, 10], atol=1e-12)
    np.testing.assert_allclose(dec["y"][1], full["y"][1, 3], atol=1e-12)
    np.testing.assert_allclose(dec["lse2"][1], full["lse2"][1, :, 3], atol=1e-12)
    assert dec["lam"] == full["lam"]


def test_grouped_ratio_one_is_v2():
    """Grouped differential attention with one signal head per noise head is
    the V2 forward (pins the head order of a group and the gate index)."""
    t = _v2_rand(seed=26, N=10)
    gate = orc.v2_gate(t["x"], t["w"])
    v2 = orc.v2_forward(t["q"], t["k"], t["v"], gate)
    gr = orc.grouped_forward(t["q"], t["k"], t["v"], gate, 1)
    np.testing.assert_allclose(gr["out"], v2["out"], atol=1e-13)


def test_grouped_gate_zero_and_shared_noise():
    """Gate 0: each output head is torch SDPA of its signal head over the
    repeated K/V (a library routine); gate 1 with every signal query equal to
    its group's noise query: exact zero; a noise head with zero query gives
    signal - gate * cumulative mean of V, the same for every signal head of
    the group."""
    r = _rng(27)
    B, N, ratio, hkv, d = 2, 9, 3, 2, 5
    Hq = 2 * (ratio + 1) * hkv  # two groups per K/V head
    q = r.standard_normal((B, N, Hq, d))
    k = r.standard_normal((B, N, hkv, d))
    v = r.standard_normal((B, N, hkv, d))
    h = Hq // (ratio + 1) * ratio
    out0 = orc.grouped_forward(q, k, v, np.zeros((B, N, h)), ratio)["out"]
    G = Hq // hkv
    kr = torch.from_numpy(np.repeat(k, G, axis=2)).permute(0, 2, 1, 3)
    vr = torch.from_numpy(np.repeat(v, G, axis=2)).permute(0, 2, 1, 3)
    sdpa = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(0, 2, 1, 3), kr, vr, is_causal=True).permute(0, 2, 1, 3).numpy()
    sig = [g * (ratio + 1) + i for g in range(Hq // (ratio + 1)) for i in range(ratio)]
    np.testing.assert_allclose(out0, sdpa[:, :, sig], atol=1e-12)
    qs = q.copy()
    for g in range(Hq // (ratio + 1)):
        for i in range(ratio):
            qs[:, :, g * (ratio + 1) + i] = q[:, :, g * (ratio + 1) + ratio]
    assert np.all(orc.grouped_forward(qs, k, v, np.ones((B, N, h)), ratio)["out"] == 0.0)
    qz = q.copy()
    qz[:, :, ratio::ratio + 1] = 0.0
    gate = r.uniform(0, 1, (B, N, h))
    got = orc.grouped_forward(qz, k, v, gate, ratio)
    cm = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None, None]
    for g in range(Hq // (ratio + 1)):
        c = (g * (ratio + 1)) // G
        for i in range(ratio):
            p = g * ratio + i
            want = sdpa[:, :, g * (ratio + 1) + i] - gate[:, :, p, None] * cm[:, :, c]
            np.testing.assert_allclose(got["out"][:, :, p], want, atol=1e-12)


# -------------------------------------------------------------- backward ----

@pytest.mark.parametrize("causal", [True, False])
def test_v1_backward_finite_differences(causal):
    """Every gradient (Q1, Q2, K1, K2, V and the four lambda vectors) against
    central differences of the forward (fp64, step 1e-6), with and without
    the causal mask."""
    t = _v1_rand(B=1, N=5, H=2, dqk=3, dv=6, seed=30, lam_std=0.4)
    li = 0.35
    r = _rng(31)
    dy = r.standard_normal((1, 5, 2, 6))
    # a non-unit RMSNorm weight on the causal case (it enters as dOhat = c w G)
    w = _rng(32).uniform(0.5, 1.5, 6) if causal else None
    grads = orc.v1_backward(t["q1"], t["q2"], t["k1"], t["k2"], t["v"], t["lq1"],
                            t["lk1"], t["lq2"], t["lk2"], li, dy, causal=causal, rms_weight=w)

    def loss(tt):
        return float(np.sum(_v1(tt, li, causal=causal, rms_weight=w)["y"] * dy))

    eps = 1e-6
    for name in ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2"):
        g = grads["d" + name]
        num = np.zeros_like(t[name])
        it = np.nditer(t[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            tp = {k: v.copy() for k, v in t.items()}
            tm = {k: v.copy() for k, v in t.items()}
            tp[name][idx] += eps
            tm[name][idx] -= eps
            num[idx] = (loss(tp) - loss(tm)) / (2 * eps)
        err = np.max(np.abs(num - g)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("causal", [True, False])
def test_v2_backward_finite_differences(causal):
    """Every V2 gradient (q, k, v, x, w_lambda) against central differences of
    gate + forward (fp64), on a GQA case with two pairs per K/V group, with
    and without the causal mask."""
    r = _rng(40)
    B, N, h, hkv, d, dm = 1, 5, 2, 1, 3, 4
    t = dict(q=r.standard_normal((B, N, 2 * h, d)), k=r.standard_normal((B, N, hkv, d)),
             v=r.standard_normal((B, N, hkv, d)), x=r.standard_normal((B, N, dm)),
             w=0.5 * r.standard_normal((dm, h)))
    dout = r.standard_normal((B, N, h, d))
    grads = orc.v2_backward(t["q"], t["k"], t["v"], t["x"], t["w"], dout, causal=causal)

    def loss(tt):
        gate = orc.v2_gate(tt["x"], tt["w"])
        return float(np.sum(orc.v2_forward(tt["q"], tt["k"], tt["v"], gate, causal=causal)["out"] * dout))

    eps = 1e-6
    for name in ("q", "k", "v", "x", "w"):
        g = grads["d" + name]
        num = np.zeros_like(t[name])
        it = np.nditer(t[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            tp = {kk: vv.copy() for kk, vv in t.items()}
            tm = {kk: vv.copy() for kk, vv in t.items()}
            tp[name][idx] += eps
            tm[name][idx] -= eps
            num[idx] = (loss(tp) - loss(tm)) / (2 * eps)
        err = np.max(np.abs(num - g)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-6, (name, err)


def test_v2_backward_gate_zero_reduces_to_even_heads():
    """With W = 0 the gate is 1/2 everywhere; with the odd queries zero the odd
    heads are uniform maps whose V-gradient is the closed form -1/2 * causal
    column means of dOut (each key j receives sum_{i >= j} dOut_i / (i + 1))."""
    r = _rng(41)
    B, N, h, hkv, d, dm = 1, 6, 1, 1, 4, 3
    q = r.standard_normal((B, N, 2, d))
    q[:, :, 1] = 0.0
    k, v = r.standard_normal((B, N, hkv, d)), r.standard_normal((B, N, hkv, d))
    x, w = r.standard_normal((B, N, dm)), np.zeros((dm, h))
    dout = r.standard_normal((B, N, h, d))
    full = orc.v2_backward(q, k, v, x, w, dout)
    s = 1 / np.sqrt(d)
    a, _ = orc.attention_maps(q[0, :, 0], k[0, :, 0], s, True)
    dv_even = a.T @ dout[0, :, 0]
    n = np.arange(1, N + 1)[:, None]
    dv_odd = -0.5 * np.cumsum((dout[0, :, 0] / n)[::-1], axis=0)[::-1]
    np.testing.assert_allclose(full["dv"][0, :, 0], dv_even + dv_odd, atol=1e-12)
    np.testing.assert_allclose(full["gate"], 0.5, atol=0)


@pytest.mark.parametrize("ratio,causal", [(3, True), (4, False), (2, True)])
def test_grouped_backward_finite_differences(ratio, causal):
    """Every grouped-attention gradient (q, k, v, x, w_lambda) against central
    differences of gate + grouped forward (fp64): two groups sharing one K/V
    head, with and without the causal mask."""
    r = _rng(50 + ratio)
    B, N, hkv, d, dm = 1, 4, 1, 3, 3
    Hq = 2 * (ratio + 1)
    h = 2 * ratio
    t = dict(q=r.standard_normal((B, N, Hq, d)), k=r.standard_normal((B, N, hkv, d)),
             v=r.standard_normal((B, N, hkv, d)), x=r.standard_normal((B, N, dm)),
             w=0.5 * r.standard_normal((dm, h)))
    dout = r.standard_normal((B, N, h, d))
    grads = orc.grouped_backward(t["q"], t["k"], t["v"], t["x"], t["w"], dout, ratio, causal=causal)

    def loss(tt):
        gate = orc.v2_gate(tt["x"], tt["w"])
        out = orc.grouped_forward(tt["q"], tt["k"], tt["v"], gate, ratio, causal=causal)["out"]
        return float(np.sum(out * dout))

    eps = 1e-6
    for name in ("q", "k", "v", "x", "w"):
        g = grads["d" + name]
        num = np.zeros_like(t[name])
        it = np.nditer(t[name], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            tp = {kk: vv.copy() for kk, vv in t.items()}
            tm = {kk: vv.copy() for kk, vv in t.items()}
            tp[name][idx] += eps
            tm[name][idx] -= eps
            num[idx] = (loss(tp) - loss(tm)) / (2 * eps)
        err = np.max(np.abs(num - g)) / max(np.max(np.abs(num)), 1e-12)
        assert err < 1e-6, (name, err)


def test_grouped_backward_ratio_one_is_v2_backward():
    """Ratio 1 (one signal head per noise head) is V2: the grouped backward
    equals the V2 backward, itself pinned by finite differences."""
    r = _rng(55)
    B, N, h, hkv, d, dm = 2, 9, 4, 2, 4, 5
    q, k, v = (r.standard_normal(s) for s in ((B, N, 2 * h, d), (B, N, hkv, d), (B, N, hkv, d)))
    x, w, dout = r.standard_normal((B, N, dm)), 0.3 * r.standard_normal((dm, h)), r.standard_normal((B, N, h, d))
    a = orc.grouped_backward(q, k, v, x, w, dout, 1)
    b = orc.v2_backward(q, k, v, x, w, dout)
    for n in ("dq", "dk", "dv", "dx", "dw", "dz"):
        np.testing.assert_allclose(a[n], b[n], rtol=1e-12, atol=1e-12 * np.max(np.abs(b[n])))


def test_grouped_backward_noise_gradient_collects_every_signal_head():
    """With the signal queries zero and the gate weight zero (every gate 1/2),
    the K/V group's dV is the closed form: the signal heads are uniform causal
    maps of dOut, the noise head a softmax map of -1/2 sum_i dOut_i, so
    dV = sum_i U^T dOut_i + A_noise^T (-1/2 sum_i dOut_i), U the uniform causal
    map (pins that every signal head of the group feeds the noise head's dO)."""
    r = _rng(56)
    ratio, B, N, d, dm = 3, 1, 6, 4, 3
    q = r.standard_normal((B, N, ratio + 1, d))
    q[:, :, :ratio] = 0.0
    k, v = r.standard_normal((B, N, 1, d)), r.standard_normal((B, N, 1, d))
    x, w = r.standard_normal((B, N, dm)), np.zeros((dm, ratio))
    dout = r.standard_normal((B, N, ratio, d))
    full = orc.grouped_backward(q, k, v, x, w, dout, ratio)
    s = 1 / np.sqrt(d)
    a_noise, _ = orc.attention_maps(q[0, :, ratio], k[0, :, 0], s, True)
    n = np.arange(1, N + 1)[:, None]
    dsum = dout[0].sum(axis=1)  # sum over the signal heads
    dv_signal = np.cumsum((dsum / n)[::-1], axis=0)[::-1]  # U^T applied to each, summed
    dv_noise = a_noise.T @ (-0.5 * dsum)
    np.testing.assert_allclose(full["dv"][0, :, 0], dv_signal + dv_noise, atol=1e-12)
