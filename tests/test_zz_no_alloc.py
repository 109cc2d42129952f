"""The V2 decode entry point that allocates nothing (diffattn_v2_decode_noalloc).

It serves callers that cannot allocate device memory (a runtime with a
fixed memory plan, a plugin that receives only inputs and outputs): its
scratch is a fixed array inside the library.  This file is collected last so
that a stop-at-first-failure run has already run every other test.  Each
check calls the entry point twice in a row (the second call reuses the
array the first one wrote) and compares both outputs with the regular
workspace entry point, within the decode parity tolerance.
"""

import ctypes as C

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 2e-2  # max|diff| <= 2e-2 * RMS(V), as for the decode parity tests


def _close(a, b, v):
    rms = float(v.float().pow(2).mean().sqrt())
    return float((a.float() - b.float()).abs().max()) <= TOL * rms


def test_noalloc_matches_workspace_entry_two_calls():
    cases = [
        dict(B=3, L=2000, h=32, hkv=8, seqlens=[2000, 1, 1333], seed=41, gate=False),
        dict(B=2, L=777, h=16, hkv=2, seqlens=[500, 777], seed=42, gate=True),
    ]
    for c in cases:  # two calls in a row, different shapes and data
        t = synth.decode_inputs(c["B"], c["L"], c["h"], c["hkv"], 128, 256, seed=c["seed"],
                                device="cuda", seqlens=c["seqlens"])
        kw = dict(seqlens=t["seqlens"])
        if c["gate"]:
            kw["gate"] = bd.diffattn_v2_gate(t["x"], t["w_lambda"])
        else:
            kw.update(x=t["x"], w_lambda=t["w_lambda"])
        ref = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], **kw)
        got = bd.diffattn_v2_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], **kw)
        torch.cuda.synchronize()
        assert _close(got, ref, t["v_cache"]), c
    assert bd.diffattn_get_device_status() == bd.DA_OK


def test_noalloc_full_decode_workload_two_calls():
    """B64, cache 32768, 64 query / 8 KV heads: the default split count is
    lowered to fit the fixed scratch; repeated calls agree with the workspace
    entry point."""
    t = synth.decode_inputs(64, 32768, 32, 8, 128, 4096, seed=1004, device="cuda")
    ref = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], x=t["x"], w_lambda=t["w_lambda"])
    for _ in range(2):
        got = bd.diffattn_v2_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], x=t["x"],
                                            w_lambda=t["w_lambda"])
        torch.cuda.synchronize()
        assert _close(got, ref, t["v_cache"][:2])
    assert bd.diffattn_get_device_status() == bd.DA_OK
    del t
    torch.cuda.empty_cache()


def test_noalloc_rejects_problems_beyond_the_fixed_scratch():
    lib = bd.load()
    p = bd.da_v2_decode_params()
    # 4096 sequences x 128 query heads x 128 features of fp32 partials even with
    # one split: 256 MiB > the fixed array
    p.B, p.h, p.h_kv, p.d, p.L_max = 4096, 64, 8, 128, 1024
    fake = torch.empty(16, dtype=torch.bfloat16, device="cuda").data_ptr()
    p.q, p.out, p.gate = fake, fake, fake
    p.k_cache = bd.da_t4(fake, 1024 * 8 * 128, 8 * 128, 128)
    p.v_cache = bd.da_t4(fake, 1024 * 8 * 128, 8 * 128, 128)
    assert lib.diffattn_v2_decode_noalloc(C.byref(p), None) == bd.DA_ERR_WORKSPACE
    # an explicit split count that does not fit is refused too
    p.B, p.num_splits = 64, 64
    assert lib.diffattn_v2_decode_noalloc(C.byref(p), None) == bd.DA_ERR_WORKSPACE
