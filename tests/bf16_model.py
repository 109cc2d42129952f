"""bf16 rounding models of the V1 and V2 backwards (test infrastructure).

Each runs the chain rule in exact fp64 EXCEPT at the points where the
library's backward must hold bf16 values.  V1: the forward outputs Y and O2,
the upstream gradient after the RMSNorm backward (dO, an MMA operand), the
P and dS tiles fed to the tensor cores, and the bf16 gradient outputs; for the
training step the forward's own P.V operand as well (``rounded_forward``).  V2: the saved per-head outputs O_j,
the odd heads' dO = -g dOut (an MMA operand), the P and dS tiles, and the
bf16 gradient outputs.  A model's error against the fp64 oracle is the error
any bf16 implementation with these storage points has; the GPU parity tests
bound the library's error by a small multiple of it.
"""

import numpy as np
import torch


def bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def rounded_forward(f, fwd, li, causal=True, rms_weight=None, eps=1e-5, rnd=bf16, scale=None):
    """The V1 forward with its own bf16 storage points, for the bars of the
    training step (the library's forward, then its backward on the forward's
    saves).  fp64 everywhere EXCEPT: P = exp(S - m) (m the row max) is rounded
    before the product with V, as the P.V operand of a bf16 tensor-core
    forward must be, while the row sum l takes the unrounded P (an fp32
    accumulation); Y = c w (O1 - lambda O2) rstd and O2 are stored rounded.
    f: fp64 inputs as in ``rounded_backward``; fwd: the oracle forward on
    them (lambda and the LSEs are taken from it).  Returns fwd with y, o2 and
    rstd replaced; with rnd the identity it reproduces the oracle forward's.
    scale: the softmax scale (None = 1/sqrt(d_qk)).  Under strong cancellation between the streams (lambda near 1, long rows)
    the rounded P dominates the step's gradient error, which the backward
    model fed exact forward outputs does not contain."""
    lam, c = fwd["lam"], 1.0 - li
    B, N, H, dqk = f["q1"].shape
    dv = f["v"].shape[3]
    s = 1.0 / np.sqrt(dqk) if scale is None else scale
    w = np.ones(dv) if rms_weight is None else rms_weight
    y = np.zeros((B, N, H, dv))
    o2 = np.zeros((B, N, H, dv))
    rstd = np.zeros((B, H, N))
    keep = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
    for b in range(B):
        for h in range(H):
            O = []
            for t in (1, 2):
                S = np.where(keep, s * f[f"q{t}"][b, :, h] @ f[f"k{t}"][b, :, h].T, -np.inf)
                P = np.exp(S - S.max(1, keepdims=True))
                O.append((rnd(P) @ f["v"][b, :, h]) / P.sum(1, keepdims=True))
            d = O[0] - lam * O[1]
            r = 1.0 / np.sqrt(np.mean(d * d, 1) + eps)
            rstd[b, h] = r
            y[b, :, h] = rnd(c * w * d * r[:, None])
            o2[b, :, h] = rnd(O[1])
    out = dict(fwd)
    out.update(y=y, o2=o2, rstd=rstd)
    return out


def _upstream(f, fw, li, b, h, rms_weight, rnd):
    """Per (batch, head): the saved Y and O2 as stored, the normalised output
    yh = Y / (c w), the RMSNorm backward's dO (an MMA operand, so stored) and
    the per-row terms <dO, O2> whose sum is -dlambda."""
    c = 1.0 - li
    Y, O2, rstd = rnd(fw["y"][b, :, h]), rnd(fw["o2"][b, :, h]), fw["rstd"][b, h]
    G = f["dy"][b, :, h]
    w = np.ones(Y.shape[1]) if rms_weight is None else rms_weight
    yh = Y / (c * w)
    gw = G * w
    gy = (gw * yh).sum(1, keepdims=True)
    dO = rnd(c * rstd[:, None] * (gw - yh * gy / Y.shape[1]))
    return dO, O2, yh, rstd, (dO * O2).sum(1)


def rounded_backward(f, fwd, li, heads=None, causal=True, rms_weight=None, rnd=bf16, exact_fwd=None,
                     scale=None):
    """f: fp64 inputs (q1..v, dy) as [B, N, H, D]; fwd: the forward on them
    (the oracle's, or ``rounded_forward``'s for the training step).  Returns
    the gradients dq1, dq2, dk1, dk2, dv and dlam computed with the bf16
    storage points (rnd; the identity gives the oracle's chain rule): the
    saved Y and O2, dO, the MMA operands dS and P, and the gradient outputs
    themselves (bf16 by the interface).  `heads` restricts to a list of heads;
    causal=False drops the key <= query mask; rms_weight is the forward's
    RMSNorm weight (None = unit); scale the softmax scale (None =
    1/sqrt(d_qk)).  With exact_fwd (the oracle forward) it also
    returns dlam_ss, the sum over rows of the squared differences between this
    model's per-row terms of dlam = -sum_rows <dO, O2> and the exact ones: the
    scale of dlam's error when the rows' errors have independent signs."""
    lam = fwd["lam"]
    B, N, H, dqk = f["q1"].shape
    heads = range(H) if heads is None else heads
    s = 1.0 / np.sqrt(dqk) if scale is None else scale
    out = {n: np.zeros_like(f["q1"]) for n in ("dq1", "dq2", "dk1", "dk2")}
    out["dv"] = np.zeros_like(f["v"])
    dlam = 0.0
    dlam_ss = 0.0
    for b in range(B):
        for h in heads:
            dO, O2, yh, rstd, D2 = _upstream(f, fwd, li, b, h, rms_weight, rnd)
            D1 = (dO * (yh / rstd[:, None] + lam * O2)).sum(1)
            dlam -= float(D2.sum())
            if exact_fwd is not None:
                D2x = _upstream(f, exact_fwd, li, b, h, rms_weight, lambda a: a)[4]
                dlam_ss += float(((D2 - D2x) ** 2).sum())
            dP = dO @ f["v"][b, :, h].T
            for t, (sig, D, lse) in enumerate(((1.0, D1, fwd["lse1"]), (-lam, D2, fwd["lse2"])), 1):
                Q, K = f[f"q{t}"][b, :, h], f[f"k{t}"][b, :, h]
                P = np.exp(s * Q @ K.T - lse[b, h][:, None])
                if causal:
                    P = np.tril(P)
                dS = rnd(sig * s * P * (dP - D[:, None]))
                out[f"dq{t}"][b, :, h] = dS @ K
                out[f"dk{t}"][b, :, h] = dS.T @ Q
                # the dV operand is P itself; sigma multiplies the stream's
                # fp32 accumulator when the streams are summed
                out["dv"][b, :, h] += sig * (rnd(P).T @ dO)
    for n in ("dq1", "dq2", "dk1", "dk2", "dv"):
        out[n] = rnd(out[n])
    out["dlam"] = dlam
    if exact_fwd is not None:
        out["dlam_ss"] = dlam_ss
    return out


def rounded_backward_v2(f, fwd, gate, scale=None, rnd=bf16, causal=True):
    """f: fp64 V2 inputs (q, k, v, x, w_lambda, dout); fwd: the oracle's V2
    forward on them; gate: fp64 [B, N, h].  Returns dq, dk, dv, dz, dx, dw
    with the V2 backward's bf16 storage points (``rnd`` = the rounding; the
    identity gives the exact chain rule)."""
    q, k, v, dout = f["q"], f["k"], f["v"], f["dout"]
    B, N, H2, d = q.shape
    group = H2 // k.shape[2]
    s = 1.0 / np.sqrt(d) if scale is None else scale
    o = rnd(fwd["o"])
    dodd = rnd(-gate[..., None] * dout)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v))
    for b in range(B):
        for j in range(H2):
            c = j // group
            dO = dout[b, :, j // 2] if j % 2 == 0 else dodd[b, :, j // 2]
            D = (dO * o[b, :, j]).sum(1)
            P = np.exp(s * q[b, :, j] @ k[b, :, c].T - fwd["lse"][b, j][:, None])
            if causal:
                P = np.tril(P)
            dS = rnd(s * P * (dO @ v[b, :, c].T - D[:, None]))
            out["dq"][b, :, j] = dS @ k[b, :, c]
            out["dk"][b, :, c] += dS.T @ q[b, :, j]
            out["dv"][b, :, c] += rnd(P).T @ dO
    dz = -(dout * o[:, :, 1::2]).sum(-1) * gate * (1.0 - gate)
    out["dz"] = dz
    out["dx"] = rnd(dz @ f["w_lambda"].T)
    out["dw"] = np.einsum("btk,btp->kp", f["x"], dz)
    for n in ("dq", "dk", "dv"):
        out[n] = rnd(out[n])
    return out


def rounded_backward_grouped(f, fwd, gate, ratio, scale=None, rnd=bf16, causal=True):
    """The grouped backward with its bf16 storage points: the saved per-head
    outputs O_j, each noise head's dO = -sum_i g_i dOut_i (summed exactly,
    rounded once), the P and dS tiles, and the bf16 gradient outputs.  f: fp64
    inputs (q, k, v, x, w_lambda, dout); fwd: the oracle's grouped forward on
    them; gate: fp64 [B, N, h].  ratio 1 gives ``rounded_backward_v2``."""
    q, k, v, dout = f["q"], f["k"], f["v"], f["dout"]
    B, N, Hq, d = q.shape
    group = Hq // k.shape[2]
    n_groups = Hq // (ratio + 1)
    s = 1.0 / np.sqrt(d) if scale is None else scale
    o = rnd(fwd["o"])
    do = np.zeros_like(o)
    dz = np.zeros_like(gate)
    for gi in range(n_groups):
        noise = gi * (ratio + 1) + ratio
        acc = np.zeros_like(dout[:, :, 0])
        for i in range(ratio):
            p = gi * ratio + i
            do[:, :, gi * (ratio + 1) + i] = dout[:, :, p]
            acc -= gate[:, :, p, None] * dout[:, :, p]
            dz[:, :, p] = -(dout[:, :, p] * o[:, :, noise]).sum(-1) * gate[:, :, p] * (1.0 - gate[:, :, p])
        do[:, :, noise] = rnd(acc)
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v))
    for b in range(B):
        for j in range(Hq):
            c = j // group
            dO = do[b, :, j]
            D = (dO * o[b, :, j]).sum(1)
            P = np.exp(s * q[b, :, j] @ k[b, :, c].T - fwd["lse"][b, j][:, None])
            if causal:
                P = np.tril(P)
            dS = rnd(s * P * (dO @ v[b, :, c].T - D[:, None]))
            out["dq"][b, :, j] = dS @ k[b, :, c]
            out["dk"][b, :, c] += dS.T @ q[b, :, j]
            out["dv"][b, :, c] += rnd(P).T @ dO
    out["dz"] = dz
    out["dx"] = rnd(dz @ f["w_lambda"].T)
    out["dw"] = np.einsum("btk,btp->kp", f["x"], dz)
    for n in ("dq", "dk", "dv"):
        out[n] = rnd(out[n])
    return out


def rounded_grouped_forward(q, k, v, gate, ratio, scale=None, causal=True, rnd=bf16):
    """The grouped forward of one group with its bf16 storage points: each
    head's P = exp(S - m) rounded as the P.V operand (the row sum from the
    unrounded P), each head's normalised output stored rounded (the o_heads
    save the combine reads), and out = O_signal - gate O_noise rounded.
    q: [N, ratio + 1, d] (signal heads, then the noise head); k, v: [N, d];
    gate: [N, ratio].  Returns out [N, ratio, d]; with rnd the identity it is
    the oracle's grouped forward of the group."""
    N, _, d = q.shape
    s = 1.0 / np.sqrt(d) if scale is None else scale
    keep = np.tril(np.ones((N, N), bool)) if causal else np.ones((N, N), bool)
    heads = []
    for j in range(ratio + 1):
        S = np.where(keep, s * q[:, j] @ k.T, -np.inf)
        P = np.exp(S - S.max(1, keepdims=True))
        heads.append(rnd((rnd(P) @ v) / P.sum(1, keepdims=True)))
    return rnd(np.stack([heads[i] - gate[:, i:i + 1] * heads[ratio] for i in range(ratio)], 1))
