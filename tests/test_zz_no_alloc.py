"""The V2 decode entry point that allocates nothing (diffattn_v2_decode_noalloc).

It serves callers that cannot allocate device memory (a runtime with a
fixed memory plan, a plugin that receives only inputs and outputs): its
scratch is a fixed array inside the library.  This file is collected last so
that a stop-at-first-failure run has already run every other test.  Each
check calls the entry point twice in a row (the second call reuses the
array the first one wrote) and compares both outputs with the regular
workspace entry point, within the decode parity tolerance; the case whose
default split count does not fit the array (so the entry point lowers it) is
also compared with the fp64 oracle, and checked to leave the device's free
memory unchanged.
"""

import ctypes as C

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from oracle import diffattn_oracle as orc

pytestmark = pytest.mark.gpu
TOL = 2e-2  # max|diff| <= 2e-2 * RMS(V), as for the decode parity tests
SCRATCH = 16 << 20  # DIFFATTN_NOALLOC_SCRATCH_BYTES


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
    """B64, cache 32768, 64 query / 8 KV heads (the decode workload): its
    partials at the default split count fit the fixed scratch as they are;
    repeated calls agree with the workspace entry point."""
    need = bd.diffattn_v2_decode_workspace_size(64, 32, 8, 128, 32768, 0, gate_given=False)
    assert need <= SCRATCH
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


def test_noalloc_lowered_split_count_against_oracle_allocates_nothing():
    """B28, cache 9216, 128 query / 8 KV heads (16 per group), gate from x:
    at the library's default split count the partials need more than the
    fixed scratch, so the entry point runs with fewer splits.  Both calls
    agree with the workspace entry point (default split count) and, on four
    whole sequences (ragged lengths included), with the fp64 oracle; the
    second call leaves the device's free memory exactly as it was."""
    B, L, h, hkv, d, dm = 28, 9216, 64, 8, 128, 256
    need = bd.diffattn_v2_decode_workspace_size(B, h, hkv, d, L, 0, gate_given=False)
    assert need > SCRATCH  # the default split count does not fit: it is lowered
    rng = np.random.default_rng(43)
    seqlens = [L] + [int(x) for x in rng.integers(1, L + 1, B - 2)] + [1]
    t = synth.decode_inputs(B, L, h, hkv, d, dm, seed=43, device="cuda", seqlens=seqlens)
    kw = dict(seqlens=t["seqlens"], x=t["x"], w_lambda=t["w_lambda"])
    ref = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], **kw)
    out = torch.empty_like(ref)
    bd.diffattn_v2_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], out=out, **kw)  # first call
    torch.cuda.synchronize()
    first = out.clone()
    free0 = torch.cuda.mem_get_info()[0]
    bd.diffattn_v2_decode_noalloc(t["q"], t["k_cache"], t["v_cache"], out=out, **kw)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.equal(out, first)  # same inputs, same split count: bit for bit
    assert _close(out, ref, t["v_cache"])
    f64 = lambda a: a.detach().to("cpu", torch.float64).numpy()  # noqa: E731
    gate = orc.v2_gate(f64(t["x"]), f64(t["w_lambda"]))
    o = f64(out)
    for b in (0, 5, 17, B - 1):
        n = seqlens[b]
        exp = orc.v2_decode(f64(t["q"][b:b + 1]), f64(t["k_cache"][b:b + 1, :n]),
                            f64(t["v_cache"][b:b + 1, :n]), [n], gate[b:b + 1])["out"][0]
        v = f64(t["v_cache"][b, :n])
        assert float(np.max(np.abs(o[b] - exp))) <= TOL * float(np.sqrt(np.mean(v * v))), b
    assert bd.diffattn_get_device_status() == bd.DA_OK
