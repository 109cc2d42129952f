"""Failure detection on the GPU without a GPU fault: a one-shot test hook
makes the V2 forward's first CTA skip one K tile load, so the waits that
depend on it expire after their ~2 s bound.  The kernel records
DA_ERR_TIMEOUT (site codes 0x2xxx belong to the V2 forward kernel) in the
device status word, the CTA's roles leave through the abort flag, and the
context stays usable: the next call is normal and correct."""

import time

import numpy as np
import pytest
import torch

from differential_attention_diff_gb300 import binding as bd
from differential_attention_diff_gb300 import synth
from oracle import diffattn_oracle as orc

pytestmark = pytest.mark.gpu


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def test_bounded_wait_expiry_is_reported_and_the_context_survives():
    t = synth.v2_inputs(1, 512, 2, 1, 128, 128, seed=91, device="cuda")
    gate = bd.diffattn_v2_gate(t["x"], t["w_lambda"])
    assert bd.diffattn_get_device_status() == bd.DA_OK
    bd.diffattn_debug_inject_fault(bd.DA_FAULT_V2_FWD_SKIP_LOAD)
    t0 = time.time()
    bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], gate=gate)
    st, raw = bd.diffattn_get_device_status(detail=True)
    elapsed = time.time() - t0
    assert st == bd.DA_ERR_TIMEOUT, (st, hex(raw))
    assert (raw >> 8) & 0xF000 == 0x2000, hex(raw)  # a V2 forward wait site
    assert 1.0 < elapsed < 30.0, elapsed             # the bound, not a hang
    # the injection was consumed: the next call runs normally and correctly
    out = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], gate=gate)
    torch.cuda.synchronize()
    assert bd.diffattn_get_device_status() == bd.DA_OK
    ref = orc.v2_forward(f64(t["q"]), f64(t["k"]), f64(t["v"]), f64(gate))
    tol = 2e-2 * float(np.sqrt(np.mean(f64(t["v"]) ** 2)))
    assert float(np.max(np.abs(f64(out) - ref["out"]))) <= tol
