"""Seeded synthetic inputs shared by the tests, the bench and the oracle legs.

This module holds no arithmetic of the method: it only draws tensors with the
shapes and distributions of the workloads (Q, K, V, X ~ N(0, 1); the four V1
lambda vectors ~ N(0, 0.1); the V2 gate weight W_lambda ~ N(0, 0.02), standard
deviations) and returns them as torch tensors.  Generation happens on the
requested device with a seeded ``torch.Generator``; callers that need the same
values on the host copy the tensors (the values, not the seed, are shared).
"""

from __future__ import annotations

import torch

_DT = {"bf16": torch.bfloat16, "f32": torch.float32}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, std, dtype, g, device):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def v1_inputs(B, N, H, dqk, dv, dtype="bf16", seed=0, device="cpu",
              with_dy=False):
    """V1 operands: q1, q2, k1, k2 [B,N,H,dqk]; v [B,N,H,dv]; four fp32 lambda
    vectors [dqk]; optionally the upstream gradient dy [B,N,H,dv]."""
    dt = _DT[dtype]
    g = _gen(seed, device)
    out = {}
    for name in ("q1", "q2", "k1", "k2"):
        out[name] = _randn((B, N, H, dqk), 1.0, dt, g, device)
    out["v"] = _randn((B, N, H, dv), 1.0, dt, g, device)
    for name in ("lq1", "lk1", "lq2", "lk2"):
        out[name] = _randn((dqk,), 0.1, torch.float32, g, device)
    if with_dy:
        out["dy"] = _randn((B, N, H, dv), 1.0, dt, g, device)
    return out


def v2_inputs(B, N, h, hkv, d, d_model, seed=0, device="cpu", with_dout=False):
    """V2 operands: q [B,N,2h,d]; k, v [B,N,hkv,d]; x [B,N,d_model];
    w_lambda [d_model,h] (all bf16); optionally the upstream gradient dout
    [B,N,h,d] ~ N(0, 1)."""
    dt = torch.bfloat16
    g = _gen(seed, device)
    out = {
        "q": _randn((B, N, 2 * h, d), 1.0, dt, g, device),
        "k": _randn((B, N, hkv, d), 1.0, dt, g, device),
        "v": _randn((B, N, hkv, d), 1.0, dt, g, device),
        "x": _randn((B, N, d_model), 1.0, dt, g, device),
        "w_lambda": _randn((d_model, h), 0.02, dt, g, device),
    }
    if with_dout:
        out["dout"] = _randn((B, N, h, d), 1.0, dt, g, device)
    return out


def grouped_inputs(B, N, h, ratio, hkv, d, d_model, seed=0, device="cpu"):
    """Grouped differential attention operands: q [B,N,h(ratio+1)/ratio,d];
    k, v [B,N,hkv,d]; x [B,N,d_model]; w_lambda [d_model,h] (all bf16)."""
    dt = torch.bfloat16
    g = _gen(seed, device)
    Hq = h // ratio * (ratio + 1)
    return {
        "q": _randn((B, N, Hq, d), 1.0, dt, g, device),
        "k": _randn((B, N, hkv, d), 1.0, dt, g, device),
        "v": _randn((B, N, hkv, d), 1.0, dt, g, device),
        "x": _randn((B, N, d_model), 1.0, dt, g, device),
        "w_lambda": _randn((d_model, h), 0.02, dt, g, device),
    }


def v1_decode_inputs(B, L_max, H, dqk, dv, seed=0, device="cpu", seqlens=None):
    """V1 decode operands: q1, q2 [B,H,dqk]; k1_cache, k2_cache [B,L_max,H,dqk];
    v_cache [B,L_max,H,dv] (bf16); four fp32 lambda vectors [dqk] ~ N(0, 0.1);
    seqlens int32 [B] (default: every sequence full)."""
    dt = torch.bfloat16
    g = _gen(seed, device)
    out = {
        "q1": _randn((B, H, dqk), 1.0, dt, g, device),
        "q2": _randn((B, H, dqk), 1.0, dt, g, device),
        "k1_cache": _randn((B, L_max, H, dqk), 1.0, dt, g, device),
        "k2_cache": _randn((B, L_max, H, dqk), 1.0, dt, g, device),
        "v_cache": _randn((B, L_max, H, dv), 1.0, dt, g, device),
    }
    for name in ("lq1", "lk1", "lq2", "lk2"):
        out[name] = _randn((dqk,), 0.1, torch.float32, g, device)
    if seqlens is None:
        seqlens = [L_max] * B
    out["seqlens"] = torch.tensor(list(seqlens), dtype=torch.int32, device=device)
    return out


def decode_inputs(B, L_max, h, hkv, d, d_model, seed=0, device="cpu",
                  seqlens=None):
    """V2 decode operands: q [B,2h,d]; k_cache, v_cache [B,L_max,hkv,d];
    x [B,d_model]; w_lambda [d_model,h] (bf16); seqlens int32 [B]
    (default: every sequence full)."""
    dt = torch.bfloat16
    g = _gen(seed, device)
    out = {
        "q": _randn((B, 2 * h, d), 1.0, dt, g, device),
        "k_cache": _randn((B, L_max, hkv, d), 1.0, dt, g, device),
        "v_cache": _randn((B, L_max, hkv, d), 1.0, dt, g, device),
        "x": _randn((B, d_model), 1.0, dt, g, device),
        "w_lambda": _randn((d_model, h), 0.02, dt, g, device),
    }
    if seqlens is None:
        seqlens = [L_max] * B
    out["seqlens"] = torch.tensor(list(seqlens), dtype=torch.int32,
                                  device=device)
    return out
