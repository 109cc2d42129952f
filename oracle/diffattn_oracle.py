"""fp64 CPU oracle for the differential-attention operator.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``differential_attention_diff_gb300/csrc``) and
imports nothing from that package.

Every function is the plain definition written out in float64 numpy: explicit
score matrices, a two-pass softmax per row (max, then exp and sum), no tiling,
no online rescaling, no fusion.  Matrix products (``@``) are the only library
primitive used as a step.

Sources (two web pages on the method; titles and sections as printed):

* [P1] "Differential Transformer | ICLR 2025 Oral" (dainus.ai blog)
  - "Softmax 어텐션의 구조적 한계": softmax rows are non-negative, sum to 1.
  - "Differential Attention: 빼기의 힘": the V1 formula
    DiffAttn(X) = (softmax(Q1 K1^T/sqrt d) - lambda softmax(Q2 K2^T/sqrt d)) V.
  - "λ의 역할과 학습": lambda_init = 0.8 - 0.6 exp(-0.3 (l - 1)).
* [P2] "Differential Transformer V2" (pogovet.com summary)
  - §1 "DIFF V1에서 V2로 바뀐 핵심 구조": V1's global lambda from dot products
    of learnable vectors plus the per-layer init, per-head RMS normalisation,
    a re-multiplied per-layer scale, V head dim twice the Q/K head dim; V2 runs
    one attention over 2h query heads, splits even/odd heads, subtracts the
    second output scaled by a sigmoid of a per-token per-head projection of X,
    and the two subtracted heads share K and V (same GQA group).
  - §3 / §4: context-RMS bounds [1/sqrt n, 1) and (0, sqrt 2).

Readings where the pages are silent (each also listed in the design notes):
the exact lambda form exp(lq1.lk1) - exp(lq2.lk2) + lambda_init, the
(1 - lambda_init) post-norm scale, RMSNorm eps 1e-5 inside the root over the
V head dim with a fixed per-feature weight (unit unless given; it takes no
gradient), 1/sqrt(d) with d the Q/K head dim, causal j <= i (or no mask),
even head 2p minus gate times odd head 2p+1, contiguous GQA groups
(q head j -> kv head j // (2h/h_kv)), no gate bias, no clamp on lambda.

Parity pins: every function here is pinned by ``tests/test_oracle.py``
(closed forms, library SDPA special cases, Hadamard-exact RMS bounds, finite
differences for the backward, decode == last causal row for V1 and V2).  None
is unpinned.

Layouts: Q/K/V are ``[B, N, H, D]`` float64 arrays (the exact bf16 / fp32
values the GPU reads, widened); per-row statistics are ``[B, H, N]``.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "lambda_init",
    "lambda_full",
    "attention_maps",
    "v1_forward",
    "v1_backward",
    "v2_gate",
    "v2_forward",
    "v2_decode",
    "v2_backward",
    "v1_decode",
    "grouped_forward",
    "grouped_backward",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def lambda_init(layer: int) -> float:
    """[P1] "λ의 역할과 학습": lambda_init(l) = 0.8 - 0.6 * exp(-0.3 * (l - 1)).

    ``layer`` is 1-based (the "(l-1)" makes l = 1 the first layer, value 0.2).
    """
    return 0.8 - 0.6 * np.exp(-0.3 * (float(layer) - 1.0))


def lambda_full(lq1, lk1, lq2, lk2, lam_init: float) -> float:
    """[P2] §1: V1's global coefficient, built from dot products of four
    learnable vectors plus the per-layer init.  Reading taken for the exact
    form: lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init, one scalar
    per layer shared by all heads; no clamp ([P1] question 1 allows lambda > 1
    and negative weights)."""
    a = float(np.dot(_f64(lq1), _f64(lk1)))
    b = float(np.dot(_f64(lq2), _f64(lk2)))
    return float(np.exp(a) - np.exp(b) + lam_init)


def attention_maps(q, k, scale: float, causal: bool, rows=None):
    """Row-softmax attention map of one head ([P1] "Softmax 어텐션의 구조적 한계").

    q: [Nq, d] queries, k: [Nk, d] keys.  Returns (A, lse) with
    A[r, j] = softmax_j(scale * <q[rows[r]], k[j]>) over the allowed keys
    (causal: j <= rows[r]; the query index and key index share one axis) and
    lse[r] = log sum_j exp(scale * <q, k_j>).  Two passes per row: the row max,
    then exponentials and their sum.
    """
    q = _f64(q)
    k = _f64(k)
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    s = scale * (q[rows] @ k.T)  # [R, Nk]
    if causal:
        keys = np.arange(k.shape[0])
        s = np.where(keys[None, :] <= rows[:, None], s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    z = e.sum(axis=1, keepdims=True)
    a = e / z
    lse = (m + np.log(z))[:, 0]
    return a, lse


def v1_forward(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, lam_init: float, *,
               scale: float | None = None, causal: bool = True,
               eps: float = 1e-5, rows=None, rms_weight=None):
    """V1 differential attention forward, then per-head RMSNorm and scale.

    [P1] "Differential Attention: 빼기의 힘":
        O = (softmax(s Q1 K1^T) - lambda softmax(s Q2 K2^T)) V,  s = 1/sqrt(d_qk)
    [P2] §1: per-head RMS normalisation after the subtraction, then the scale
    given by the per-layer init, read as
        Y = (1 - lambda_init) * w * O / sqrt(mean_k O_k^2 + eps)
    over the V head dim (2 d_qk) of each (b, n, h); w is the RMSNorm weight
    ([d_v], shared by heads; None = unit, as the pages' configuration).

    q1, q2, k1, k2: [B, N, H, d_qk]; v: [B, N, H, d_v]; lq1..lk2: [d_qk].
    ``rows`` restricts the query rows computed (every key is still used).
    Returns a dict: y, o (pre-norm), o2 (= A2 V), lse1, lse2, rstd ([B,H,R]),
    lam (the scalar), rows.
    """
    q1, q2, k1, k2, v = (_f64(t) for t in (q1, q2, k1, k2, v))
    B, N, H, dqk = q1.shape
    dv = v.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    lam = lambda_full(lq1, lk1, lq2, lk2, lam_init)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    R = rows.shape[0]
    y = np.zeros((B, R, H, dv))
    o = np.zeros((B, R, H, dv))
    o2 = np.zeros((B, R, H, dv))
    lse1 = np.zeros((B, H, R))
    lse2 = np.zeros((B, H, R))
    rstd = np.zeros((B, H, R))
    c = 1.0 - lam_init
    w = np.ones(dv) if rms_weight is None else _f64(rms_weight)
    for b in range(B):
        for h in range(H):
            a1, l1 = attention_maps(q1[b, :, h], k1[b, :, h], scale, causal, rows)
            a2, l2 = attention_maps(q2[b, :, h], k2[b, :, h], scale, causal, rows)
            o_bh = (a1 - lam * a2) @ v[b, :, h]
            o2_bh = a2 @ v[b, :, h]
            r = np.sqrt(np.mean(o_bh * o_bh, axis=1) + eps)
            y[b, :, h] = c * w * o_bh / r[:, None]
            o[b, :, h] = o_bh
            o2[b, :, h] = o2_bh
            lse1[b, h] = l1
            lse2[b, h] = l2
            rstd[b, h] = 1.0 / r
    return dict(y=y, o=o, o2=o2, lse1=lse1, lse2=lse2, rstd=rstd, lam=lam,
                rows=rows)


def v1_backward(q1, q2, k1, k2, v, lq1, lk1, lq2, lk2, lam_init: float, dy, *,
                scale: float | None = None, causal: bool = True,
                eps: float = 1e-5, rms_weight=None):
    """Gradients of the V1 forward above (all rows), by the chain rule.

    The pages give no backward formulas; this is the derivative of
    ``v1_forward`` written step by step.  With c = 1 - lambda_init, w the
    RMSNorm weight (a constant: no gradient), r = sqrt(mean O^2 + eps),
    Ohat = O / r, G = dY:
      dOhat = c w G;  dO = (dOhat - Ohat * mean(dOhat * Ohat)) / r
      dlambda = -sum <dO, A2 V>
      dP = dO V^T
      dS1 = A1 * (dP - <dO, A1 V>),  dS2 = -lambda A2 * (dP - <dO, A2 V>)
      dQt = s dSt Kt,  dKt = s dSt^T Qt,  dV = (A1 - lambda A2)^T dO
      lambda = e^a - e^b + lambda_init, a = lq1.lk1, b = lq2.lk2:
      dlq1 = dlambda e^a lk1, dlk1 = dlambda e^a lq1,
      dlq2 = -dlambda e^b lk2, dlk2 = -dlambda e^b lq2.
    Pinned against central finite differences of ``v1_forward``.
    """
    q1, q2, k1, k2, v, dy = (_f64(t) for t in (q1, q2, k1, k2, v, dy))
    lq1, lk1, lq2, lk2 = (_f64(t) for t in (lq1, lk1, lq2, lk2))
    B, N, H, dqk = q1.shape
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    lam = lambda_full(lq1, lk1, lq2, lk2, lam_init)
    c = 1.0 - lam_init
    w = np.ones(v.shape[-1]) if rms_weight is None else _f64(rms_weight)
    grads = {name: np.zeros_like(t) for name, t in
             (("dq1", q1), ("dq2", q2), ("dk1", k1), ("dk2", k2), ("dv", v))}
    dlam = 0.0
    for b in range(B):
        for h in range(H):
            Q1, Q2, K1, K2, V = (t[b, :, h] for t in (q1, q2, k1, k2, v))
            a1, _ = attention_maps(Q1, K1, scale, causal)
            a2, _ = attention_maps(Q2, K2, scale, causal)
            O = (a1 - lam * a2) @ V
            O2 = a2 @ V
            O1 = a1 @ V
            r = np.sqrt(np.mean(O * O, axis=1) + eps)
            Ohat = O / r[:, None]
            dOhat = c * w * dy[b, :, h]
            dO = (dOhat - Ohat * np.mean(dOhat * Ohat, axis=1, keepdims=True)) / r[:, None]
            dlam += -float(np.sum(dO * O2))
            dP = dO @ V.T
            D1 = np.sum(dO * O1, axis=1, keepdims=True)
            D2 = np.sum(dO * O2, axis=1, keepdims=True)
            dS1 = a1 * (dP - D1)
            dS2 = -lam * a2 * (dP - D2)
            grads["dq1"][b, :, h] = scale * dS1 @ K1
            grads["dq2"][b, :, h] = scale * dS2 @ K2
            grads["dk1"][b, :, h] = scale * dS1.T @ Q1
            grads["dk2"][b, :, h] = scale * dS2.T @ Q2
            grads["dv"][b, :, h] = (a1 - lam * a2).T @ dO
    ea = np.exp(np.dot(lq1, lk1))
    eb = np.exp(np.dot(lq2, lk2))
    grads["dlq1"] = dlam * ea * lk1
    grads["dlk1"] = dlam * ea * lq1
    grads["dlq2"] = -dlam * eb * lk2
    grads["dlk2"] = -dlam * eb * lq2
    grads["dlam"] = dlam
    grads["lam"] = lam
    return grads


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def v2_gate(x, w):
    """[P2] §1 / §4: per-token, per-head coefficient projected from the input X
    and passed through a sigmoid: g[..., p] = sigmoid(sum_k X[..., k] W[k, p]).
    No bias (the pages name none)."""
    return _sigmoid(_f64(x) @ _f64(w))


def v2_forward(q, k, v, gate, *, scale: float | None = None,
               causal: bool = True, rows=None):
    """V2 differential attention forward ([P2] §1, one-line summary, §8).

    One attention over 2h query heads with h_kv K/V heads (GQA, contiguous
    groups: q head j reads kv head j // (2h / h_kv)); the per-head outputs are
    split into even and odd heads and combined per token and pair p as
        Out[b, t, p] = O[b, t, 2p] - gate[b, t, p] * O[b, t, 2p + 1].
    No normalisation afterwards ([P2] §4 removes V1's RMSNorm).

    q: [B, N, 2h, d]; k, v: [B, N, h_kv, d]; gate: [B, N, h].
    Returns dict: out [B, R, h, d], o (per q head) [B, R, 2h, d], lse [B, 2h, R].
    """
    q, k, v, gate = (_f64(t) for t in (q, k, v, gate))
    B, N, H2, d = q.shape
    hkv = k.shape[2]
    group = H2 // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    R = rows.shape[0]
    o = np.zeros((B, R, H2, d))
    lse = np.zeros((B, H2, R))
    for b in range(B):
        for j in range(H2):
            g = j // group
            a, l = attention_maps(q[b, :, j], k[b, :, g], scale, causal, rows)
            o[b, :, j] = a @ v[b, :, g]
            lse[b, j] = l
    out = o[:, :, 0::2] - gate[:, rows, :, None] * o[:, :, 1::2]
    return dict(out=out, o=o, lse=lse, rows=rows)


def v2_backward(q, k, v, x, w, dout, *, scale: float | None = None, causal: bool = True):
    """Gradients of the V2 forward (``v2_gate`` then ``v2_forward``) with
    respect to q, k, v, x and w, given dOut.  The pages state no backward; this
    is the chain rule of the forward above, step by step.  With g = sigmoid(z),
    z = X W, Out_p = O_2p - g_p O_2p+1, G = dOut:
      dO_2p = G,  dO_2p+1 = -g G,  dg_p = -<G_p, O_2p+1>,  dz = dg g (1 - g)
      dW = X^T dz,  dX = dz W^T
      per query head j (kv head c = j // group):  A = softmax(s Q_j K_c^T),
      dP = dO_j V_c^T,  dS = A * (dP - <dO_j, O_j>),
      dQ_j = s dS K_c,  dK_c += s dS^T Q_j,  dV_c += A^T dO_j.
    Pinned against central finite differences of the forward."""
    q, k, v, x, w, dout = (_f64(t) for t in (q, k, v, x, w, dout))
    B, N, H2, d = q.shape
    hkv = k.shape[2]
    group = H2 // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    z = x @ w
    g = _sigmoid(z)
    fwd = v2_forward(q, k, v, g, scale=scale, causal=causal)
    o = fwd["o"]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    do = np.zeros_like(o)
    do[:, :, 0::2] = dout
    do[:, :, 1::2] = -g[..., None] * dout
    dg = -np.sum(dout * o[:, :, 1::2], axis=-1)
    dz = dg * g * (1.0 - g)
    dw = np.einsum("btk,btp->kp", x, dz)
    dx = dz @ w.T
    for b in range(B):
        for j in range(H2):
            c = j // group
            Q, K, V = q[b, :, j], k[b, :, c], v[b, :, c]
            a, _ = attention_maps(Q, K, scale, causal)
            dO = do[b, :, j]
            dP = dO @ V.T
            D = np.sum(dO * o[b, :, j], axis=1, keepdims=True)
            dS = a * (dP - D)
            dq[b, :, j] = scale * dS @ K
            dk[b, :, c] += scale * dS.T @ Q
            dv[b, :, c] += a.T @ dO
    return dict(dq=dq, dk=dk, dv=dv, dx=dx, dw=dw, dz=dz, gate=g, o=o, lse=fwd["lse"])


def v2_decode(q, k_cache, v_cache, seqlens, gate, *, scale: float | None = None):
    """V2 decode ([P1] "V2로의 진화", [P2] §2): one new token per sequence
    attends over the first seqlens[b] cached positions (the new token's own
    K/V is already in the cache at position seqlens[b] - 1), then the even /
    odd combination with the per-token per-head gate.

    q: [B, 2h, d]; k_cache, v_cache: [B, L_max, h_kv, d]; seqlens: [B] ints;
    gate: [B, h].  Returns dict: out [B, h, d], o [B, 2h, d], lse [B, 2h].
    """
    q, k_cache, v_cache, gate = (_f64(t) for t in (q, k_cache, v_cache, gate))
    B, H2, d = q.shape
    hkv = k_cache.shape[2]
    group = H2 // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    o = np.zeros((B, H2, d))
    lse = np.zeros((B, H2))
    for b in range(B):
        L = int(seqlens[b])
        for j in range(H2):
            g = j // group
            a, l = attention_maps(q[b, j][None, :], k_cache[b, :L, g], scale,
                                  causal=False)
            o[b, j] = a[0] @ v_cache[b, :L, g]
            lse[b, j] = l[0]
    out = o[:, 0::2] - gate[:, :, None] * o[:, 1::2]
    return dict(out=out, o=o, lse=lse)


def v1_decode(q1, q2, k1_cache, k2_cache, v_cache, seqlens, lq1, lk1, lq2, lk2,
              lam_init: float, *, scale: float | None = None, eps: float = 1e-5,
              rms_weight=None):
    """V1 decode: one new token per sequence, the V1 operator of [P1]
    "Differential Attention: 빼기의 힘" (two maps over two K caches, one shared
    V cache) followed by the per-head RMSNorm and (1 - lambda_init) scale of
    [P2] §1, for the query of the token at position seqlens[b] - 1 (its own
    K1/K2/V rows are already in the caches).  [P1] "V2로의 진화" names LLM
    decoding as the memory-bound case.

    q1, q2: [B, H, d_qk]; k1_cache, k2_cache: [B, L_max, H, d_qk];
    v_cache: [B, L_max, H, d_v]; seqlens: [B] ints; rms_weight: [d_v] or
    None (unit), as in ``v1_forward``.
    Returns dict: y [B, H, d_v], o (pre-norm) [B, H, d_v], lse1, lse2 [B, H],
    lam.
    """
    q1, q2, k1_cache, k2_cache, v_cache = (_f64(t) for t in (q1, q2, k1_cache, k2_cache, v_cache))
    B, H, dqk = q1.shape
    dv = v_cache.shape[-1]
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    lam = lambda_full(lq1, lk1, lq2, lk2, lam_init)
    c = 1.0 - lam_init
    w = np.ones(dv) if rms_weight is None else _f64(rms_weight)
    y = np.zeros((B, H, dv))
    o = np.zeros((B, H, dv))
    lse1 = np.zeros((B, H))
    lse2 = np.zeros((B, H))
    for b in range(B):
        L = int(seqlens[b])
        for h in range(H):
            a1, l1 = attention_maps(q1[b, h][None, :], k1_cache[b, :L, h], scale, causal=False)
            a2, l2 = attention_maps(q2[b, h][None, :], k2_cache[b, :L, h], scale, causal=False)
            o_bh = ((a1 - lam * a2) @ v_cache[b, :L, h])[0]
            r = np.sqrt(np.mean(o_bh * o_bh) + eps)
            y[b, h] = c * w * o_bh / r
            o[b, h] = o_bh
            lse1[b, h] = l1[0]
            lse2[b, h] = l2[0]
    return dict(y=y, o=o, lse1=lse1, lse2=lse2, lam=lam)


def grouped_forward(q, k, v, gate, ratio: int, *, scale: float | None = None,
                    causal: bool = True, rows=None):
    """Grouped differential attention, forward.  [P1] "같은 문제, 다른 접근"
    names it as a follow-up that gives signal heads and noise heads an uneven
    share, 3:1 or 4:1; the pages give nothing more.  Plainest reading, in the
    V2 form ([P2] §1: one GQA attention, the subtracted heads share K and V,
    a per-token per-head sigmoid gate): the query heads come in groups of
    ``ratio`` signal heads followed by one noise head, and every signal head
    subtracts the gated output of its group's noise head:
        Out[b, t, g r + i] = O[b, t, g (r+1) + i]
                             - gate[b, t, g r + i] * O[b, t, g (r+1) + r]
    for i < r.  With ratio 1 this is the V2 forward exactly.

    q: [B, N, h (r+1) / r, d]; k, v: [B, N, h_kv, d] (contiguous GQA groups,
    each holding whole signal/noise groups); gate: [B, N, h].
    ``rows`` restricts the query rows computed (every key is still used).
    Returns dict: out [B, R, h, d], o (per query head) [B, R, Hq, d],
    lse [B, Hq, R], rows.
    """
    q, k, v, gate = (_f64(t) for t in (q, k, v, gate))
    B, N, Hq, d = q.shape
    hkv = k.shape[2]
    group = Hq // hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    R = rows.shape[0]
    o = np.zeros((B, R, Hq, d))
    lse = np.zeros((B, Hq, R))
    for b in range(B):
        for j in range(Hq):
            c = j // group
            a, l = attention_maps(q[b, :, j], k[b, :, c], scale, causal, rows)
            o[b, :, j] = a @ v[b, :, c]
            lse[b, j] = l
    n_groups = Hq // (ratio + 1)
    h = n_groups * ratio
    out = np.zeros((B, R, h, d))
    for g in range(n_groups):
        noise = o[:, :, g * (ratio + 1) + ratio]
        for i in range(ratio):
            p = g * ratio + i
            out[:, :, p] = o[:, :, g * (ratio + 1) + i] - gate[:, rows, p, None] * noise
    return dict(out=out, o=o, lse=lse, rows=rows)


def grouped_backward(q, k, v, x, w, dout, ratio: int, *, scale: float | None = None,
                     causal: bool = True):
    """Gradients of grouped differential attention (``v2_gate`` then
    ``grouped_forward``) with respect to q, k, v, x and w, given dOut.  The
    pages state no backward ([P1] "같은 문제, 다른 접근" names the 3:1 / 4:1
    signal:noise follow-up only); this is the chain rule of the forward above,
    step by step.  With r = ratio, group gi holding signal heads
    gi (r+1) + i (i < r) and noise head gi (r+1) + r, output head
    p = gi r + i, g = sigmoid(z), z = X W, G = dOut:
      Out_p = O_signal(p) - g_p O_noise(gi)
      dO_signal(p) = G_p,   dO_noise(gi) = -sum_i g_p G_p
      dg_p = -<G_p, O_noise(gi)>,   dz = dg g (1 - g)
      dW = X^T dz,  dX = dz W^T
      per query head j (kv head c = j // group):  A = softmax(s Q_j K_c^T),
      dP = dO_j V_c^T,  dS = A * (dP - <dO_j, O_j>),
      dQ_j = s dS K_c,  dK_c += s dS^T Q_j,  dV_c += A^T dO_j.
    Pinned against central finite differences of the forward, and against
    ``v2_backward`` at ratio 1."""
    q, k, v, x, w, dout = (_f64(t) for t in (q, k, v, x, w, dout))
    B, N, Hq, d = q.shape
    hkv = k.shape[2]
    group = Hq // hkv
    n_groups = Hq // (ratio + 1)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    z = x @ w
    g = _sigmoid(z)
    fwd = grouped_forward(q, k, v, g, ratio, scale=scale, causal=causal)
    o = fwd["o"]
    do = np.zeros_like(o)
    dg = np.zeros_like(g)
    for gi in range(n_groups):
        noise = gi * (ratio + 1) + ratio
        for i in range(ratio):
            p = gi * ratio + i
            do[:, :, gi * (ratio + 1) + i] = dout[:, :, p]
            do[:, :, noise] -= g[:, :, p, None] * dout[:, :, p]
            dg[:, :, p] = -np.sum(dout[:, :, p] * o[:, :, noise], axis=-1)
    dz = dg * g * (1.0 - g)
    dw = np.einsum("btk,btp->kp", x, dz)
    dx = dz @ w.T
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for j in range(Hq):
            c = j // group
            Q, K, V = q[b, :, j], k[b, :, c], v[b, :, c]
            a, _ = attention_maps(Q, K, scale, causal)
            dO = do[b, :, j]
            dP = dO @ V.T
            D = np.sum(dO * o[b, :, j], axis=1, keepdims=True)
            dS = a * (dP - D)
            dq[b, :, j] = scale * dS @ K
            dk[b, :, c] += scale * dS.T @ Q
            dv[b, :, c] += a.T @ dO
    return dict(dq=dq, dk=dk, dv=dv, dx=dx, dw=dw, dz=dz, gate=g, o=o, lse=fwd["lse"])
