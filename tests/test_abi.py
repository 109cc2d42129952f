"""Host-side checks of the C ABI: the library loads without a GPU, exports
every entry point that include/diffattn.h declares, and rejects bad
arguments before launching anything."""

import ctypes as C
import math
import os
import re

import pytest

from differential_attention_diff_gb300 import binding as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "diffattn.h")).read()
    return sorted(set(re.findall(r"\b(diffattn_\w+)\s*\(", src)))


def test_header_matches_binding_list():
    assert _declared() == sorted(bd.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_lambda_init_host_function(lib):
    """lambda_init(l) = 0.8 - 0.6 exp(-0.3 (l - 1)) ("Differential Transformer",
    section 'λ의 역할과 학습'); checked against the closed form in fp32."""
    assert bd.diffattn_lambda_init(1) == pytest.approx(0.2, abs=1e-7)
    for l in (2, 5, 14, 28):
        assert bd.diffattn_lambda_init(l) == pytest.approx(0.8 - 0.6 * math.exp(-0.3 * (l - 1)), abs=1e-7)
    assert math.isnan(bd.diffattn_lambda_init(0))


def test_status_strings(lib):
    for s in range(7):
        assert lib.diffattn_status_string(s)
    assert lib.diffattn_status_string(99) == b"unknown status"


def test_null_params_rejected(lib):
    for name in ("diffattn_v1_fwd", "diffattn_v1_bwd", "diffattn_v2_gate", "diffattn_v2_fwd",
                 "diffattn_v2_decode", "diffattn_v2_decode_noalloc", "diffattn_v2_bwd", "diffattn_v1_decode",
                 "diffattn_grouped_fwd", "diffattn_grouped_bwd"):
        assert getattr(lib, name)(None, None) == bd.DA_ERR_INVALID_ARG, name


def _v1p(**kw):
    p = bd.da_v1_fwd_params()
    p.B, p.N, p.H, p.d_qk, p.d_v = 1, 64, 2, 128, 256
    p.dtype, p.causal, p.lambda_init, p.rms_eps = bd.DA_BF16, 1, 0.2, 1e-5
    fake = 1 << 20  # never dereferenced: validation fails or stops first
    for n in ("q1", "q2", "k1", "k2", "v", "out"):
        setattr(p, n, bd.da_t4(fake, 64 * 2 * 256, 2 * 256, 256))
    for n in ("lq1", "lk1", "lq2", "lk2"):
        setattr(p, n, fake)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_v1_fwd_argument_checks(lib):
    f = lib.diffattn_v1_fwd
    assert f(C.byref(_v1p(B=-1)), None) == bd.DA_ERR_INVALID_ARG
    assert f(C.byref(_v1p(dtype=7)), None) == bd.DA_ERR_INVALID_ARG
    assert f(C.byref(_v1p(lq1=None)), None) == bd.DA_ERR_INVALID_ARG
    assert f(C.byref(_v1p(q1=bd.da_t4(None, 0, 0, 0))), None) == bd.DA_ERR_INVALID_ARG
    # misaligned bf16 base pointer and a stride that is not a multiple of 8
    assert f(C.byref(_v1p(k1=bd.da_t4((1 << 20) + 2, 64, 64, 64))), None) == bd.DA_ERR_INVALID_ARG
    assert f(C.byref(_v1p(v=bd.da_t4(1 << 20, 64, 60, 64))), None) == bd.DA_ERR_INVALID_ARG
    assert f(C.byref(_v1p(rms_eps=-1.0)), None) == bd.DA_ERR_INVALID_ARG
    assert f(C.byref(_v1p(rms_weight=(1 << 20) + 2)), None) == bd.DA_ERR_INVALID_ARG  # fp32 alignment
    # empty problems are a no-op
    assert f(C.byref(_v1p(N=0)), None) == bd.DA_OK


def test_v1_bwd_causal_and_deterministic_checks(lib):
    """Causal or not, either dQ mode, is accepted (each combination reaches
    the workspace check, with none given)."""
    p = bd.da_v1_bwd_params()
    p.B, p.N, p.H, p.d_qk, p.d_v, p.dtype = 1, 256, 2, 128, 256, bd.DA_BF16
    p.lambda_init, p.rms_eps = 0.2, 1e-5
    fake = 1 << 20
    for n in ("q1", "q2", "k1", "k2", "dq1", "dq2", "dk1", "dk2"):
        setattr(p, n, bd.da_t4(fake, 1 << 16, 1 << 8, 128))
    for n in ("v", "out", "dout", "o2", "dv"):
        setattr(p, n, bd.da_t4(fake, 1 << 17, 1 << 9, 256))
    for n in ("lq1", "lk1", "lq2", "lk2", "dlq1", "dlk1", "dlq2", "dlk2", "lse1", "lse2", "rstd"):
        setattr(p, n, fake)
    f = lib.diffattn_v1_bwd
    for causal, det, want in ((1, 0, bd.DA_ERR_WORKSPACE), (0, 0, bd.DA_ERR_WORKSPACE),
                              (1, 1, bd.DA_ERR_WORKSPACE), (0, 1, bd.DA_ERR_WORKSPACE)):
        p.causal, p.deterministic = causal, det
        assert f(C.byref(p), None) == want, (causal, det)


def test_decode_argument_checks(lib):
    p = bd.da_v2_decode_params()
    p.B, p.h, p.h_kv, p.d, p.L_max = 2, 32, 8, 128, 1024
    fake = 1 << 20
    p.q, p.out, p.gate = fake, fake, fake
    p.k_cache = bd.da_t4(fake, 1024 * 8 * 128, 8 * 128, 128)
    p.v_cache = bd.da_t4(fake, 1024 * 8 * 128, 8 * 128, 128)
    f = lib.diffattn_v2_decode
    bad = bd.da_v2_decode_params.from_buffer_copy(p)
    bad.h_kv = 3  # 2h not divisible into groups
    assert f(C.byref(bad), None) == bd.DA_ERR_INVALID_ARG
    bad = bd.da_v2_decode_params.from_buffer_copy(p)
    bad.h, bad.h_kv = 4, 8  # group of one query head: a pair would straddle groups
    assert f(C.byref(bad), None) == bd.DA_ERR_INVALID_ARG
    bad = bd.da_v2_decode_params.from_buffer_copy(p)
    bad.d = 96
    assert f(C.byref(bad), None) == bd.DA_ERR_UNSUPPORTED
    bad.d = 64  # supported: the next check is the workspace
    assert f(C.byref(bad), None) == bd.DA_ERR_WORKSPACE
    # workspace missing
    assert f(C.byref(p), None) == bd.DA_ERR_WORKSPACE
    ws = lib.diffattn_v2_decode_workspace_size(2, 32, 8, 128, 1024, 4, 1)
    assert ws >= 4 * 2 * 64 * 128 * 4
    assert lib.diffattn_v2_decode_workspace_size(2, 32, 8, 128, 1024, 4, 0) > ws


def test_noalloc_decode_reports_shape_errors_before_size(lib):
    """The entry point without a workspace checks shapes as diffattn_v2_decode
    does before it sizes the partials: a malformed problem that would also be
    too large for its fixed scratch is reported as malformed, not as one that
    does not fit."""
    p = bd.da_v2_decode_params()
    p.B, p.h, p.h_kv, p.d, p.L_max = 4096, 64, 8, 128, 1024  # too large for the scratch
    fake = 1 << 20
    p.q, p.out, p.gate = fake, fake, fake
    p.k_cache = bd.da_t4(fake, 1024 * 8 * 128, 8 * 128, 128)
    p.v_cache = bd.da_t4(fake, 1024 * 8 * 128, 8 * 128, 128)
    f = lib.diffattn_v2_decode_noalloc
    for field, value, expect in (("d", 96, bd.DA_ERR_UNSUPPORTED), ("h_kv", 3, bd.DA_ERR_INVALID_ARG),
                                 ("h_kv", 128, bd.DA_ERR_INVALID_ARG), ("num_splits", 70000, bd.DA_ERR_INVALID_ARG)):
        bad = bd.da_v2_decode_params.from_buffer_copy(p)
        setattr(bad, field, value)
        assert f(C.byref(bad), None) == expect, (field, value)
        assert lib.diffattn_v2_decode(C.byref(bad), None) == expect, (field, value)


def test_v2_fwd_argument_checks(lib):
    p = bd.da_v2_fwd_params()
    p.B, p.N, p.h, p.h_kv, p.d, p.causal = 1, 128, 32, 8, 128, 1
    fake = 1 << 20
    for n in ("q", "k", "v", "out"):
        setattr(p, n, bd.da_t4(fake, 1 << 16, 1 << 10, 128))
    f = lib.diffattn_v2_fwd
    # neither a gate nor x / w_lambda
    assert f(C.byref(p), None) == bd.DA_ERR_INVALID_ARG
    p.x, p.w_lambda, p.d_model = fake, fake, 4096
    assert f(C.byref(p), None) == bd.DA_ERR_WORKSPACE
    p.d = 64   # head dim 64 is supported: the next check is the workspace
    assert f(C.byref(p), None) == bd.DA_ERR_WORKSPACE
    p.d = 96
    assert f(C.byref(p), None) == bd.DA_ERR_UNSUPPORTED
    assert lib.diffattn_v2_fwd_workspace_size(2, 8192, 32, 0) == 2 * 8192 * 32 * 4
    assert lib.diffattn_v2_fwd_workspace_size(2, 8192, 32, 1) == 0


def test_gate_argument_checks(lib):
    p = bd.da_v2_gate_params(16, 100, 32, 1 << 20, 100, 1 << 20, 1 << 20)
    assert lib.diffattn_v2_gate(C.byref(p), None) == bd.DA_ERR_INVALID_ARG  # stride % 8
    p = bd.da_v2_gate_params(16, 96, 32, 1 << 20, 96, 1 << 20, 1 << 20)
    assert lib.diffattn_v2_gate(C.byref(p), None) == bd.DA_ERR_UNSUPPORTED  # d_model % 64
    p = bd.da_v2_gate_params(0, 64, 32, None, 64, None, None)
    assert lib.diffattn_v2_gate(C.byref(p), None) == bd.DA_OK  # empty


def test_bwd_workspace_size(lib):
    base = lib.diffattn_v1_bwd_workspace_size(1, 8192, 16, 128, 256, 0)
    det = lib.diffattn_v1_bwd_workspace_size(1, 8192, 16, 128, 256, 1)
    assert base > 0 and lib.diffattn_v1_bwd_workspace_size(0, 8192, 16, 128, 256, 0) == 0
    # head dims (64, 128): dO and the dQ accumulators shrink by half (per row:
    # d_v bf16 of dO + 2 streams x d_qk fp32 = 512 -> 256 bytes)
    small = lib.diffattn_v1_bwd_workspace_size(1, 8192, 16, 64, 128, 0)
    assert base - small >= 8192 * 16 * 256
    # deterministic mode: one fp32 [64, 128] slot per (key tile, query tile)
    # pair and stream replaces the [N, 128] accumulators; the size query has no
    # mask flag, so it covers every pair (a causal call uses only the pairs
    # with query tile >= 2 key tile)
    n_kt, n_qt = 8192 // 128, 8192 // 64
    slots = n_kt * n_qt
    assert det - base == 2 * 16 * (slots * 64 - 8192) * 128 * 4
    assert lib.diffattn_v2_bwd_workspace_size(2, 8192, 32, 4096) > lib.diffattn_v2_bwd_workspace_size(2, 8192, 32, 0)


def test_v1_fwd_workspace_size(lib):
    # bf16 path: a 256-byte work counter, then one 64 KB exchange slot
    # (128 rows x 128 fp32) per CTA of every 2-CTA cluster that can run at once
    ws = lib.diffattn_v1_fwd_workspace_size(4, 4096, 12, 128, 256, bd.DA_BF16)
    slot = 128 * 128 * 4
    assert ws > 256 and (ws - 256) % (2 * slot) == 0
    # the same for the (64, 128) head dims (the slot is sized for the larger)
    assert lib.diffattn_v1_fwd_workspace_size(4, 4096, 12, 64, 128, bd.DA_BF16) == ws
    # the fp32 path needs none; empty shapes need none
    assert lib.diffattn_v1_fwd_workspace_size(1, 64, 2, 16, 32, bd.DA_F32) == 0
    assert lib.diffattn_v1_fwd_workspace_size(0, 4096, 12, 128, 256, bd.DA_BF16) == 0


def test_grouped_shape_checks(lib):
    """Grouped differential attention rejects, before any launch, groups that
    do not divide the heads or straddle K/V groups, and an odd number of query
    heads per K/V head (the attention kernel takes heads two at a time)."""
    def p(h, ratio, hkv):
        return bd.da_grouped_fwd_params(B=1, N=64, h=h, ratio=ratio, h_kv=hkv, d=128, d_model=0, causal=1)
    assert lib.diffattn_grouped_fwd(C.byref(p(7, 3, 1)), None) == bd.DA_ERR_INVALID_ARG   # h % ratio
    assert lib.diffattn_grouped_fwd(C.byref(p(6, 3, 4)), None) == bd.DA_ERR_INVALID_ARG   # 8 heads / 4 kv: groups of 4 straddle
    assert lib.diffattn_grouped_fwd(C.byref(p(8, 4, 2)), None) == bd.DA_ERR_UNSUPPORTED   # 5 heads per kv head
    assert lib.diffattn_grouped_fwd_workspace_size(2, 8192, 48, 3, 128, 0, 0) == 2 * 8192 * 48 * 4 + 2 * 8192 * 64 * 128 * 2


def test_fault_hook_arguments(lib):
    """The test hook accepts only the faults it knows, and NONE disarms it
    (host-side state: no kernel is launched)."""
    assert lib.diffattn_debug_inject_fault(7) == bd.DA_ERR_INVALID_ARG
    assert lib.diffattn_debug_inject_fault(bd.DA_FAULT_V2_FWD_SKIP_LOAD) == bd.DA_OK
    assert lib.diffattn_debug_inject_fault(bd.DA_FAULT_NONE) == bd.DA_OK


def test_v1_decode_argument_checks(lib):
    p = bd.da_v1_decode_params()
    p.B, p.H, p.d_qk, p.d_v, p.L_max = 2, 4, 128, 256, 1024
    p.lambda_init, p.rms_eps = 0.2, 1e-5
    fake = 1 << 20
    p.q1, p.q2, p.out = fake, fake, fake
    p.lq1 = p.lk1 = p.lq2 = p.lk2 = fake
    p.k1_cache = bd.da_t4(fake, 1024 * 4 * 128, 4 * 128, 128)
    p.k2_cache = bd.da_t4(fake, 1024 * 4 * 128, 4 * 128, 128)
    p.v_cache = bd.da_t4(fake, 1024 * 4 * 256, 4 * 256, 256)
    f = lib.diffattn_v1_decode

    def with_(**kw):
        q = bd.da_v1_decode_params.from_buffer_copy(p)
        for k, v in kw.items():
            setattr(q, k, v)
        return C.byref(q)
    assert f(with_(d_qk=64), None) == bd.DA_ERR_UNSUPPORTED              # d_v must be 2 d_qk
    assert f(with_(d_qk=64, d_v=128), None) == bd.DA_ERR_WORKSPACE        # supported head dims
    assert f(with_(d_qk=96, d_v=192), None) == bd.DA_ERR_UNSUPPORTED
    assert f(with_(q1=fake + 2), None) == bd.DA_ERR_INVALID_ARG          # misaligned query
    assert f(with_(lk2=None), None) == bd.DA_ERR_INVALID_ARG
    assert f(with_(rms_eps=-1.0), None) == bd.DA_ERR_INVALID_ARG
    assert f(with_(v_cache=bd.da_t4(fake, 1024, 12, 256)), None) == bd.DA_ERR_INVALID_ARG  # stride % 8
    assert f(with_(num_splits=70000), None) == bd.DA_ERR_INVALID_ARG
    assert f(with_(), None) == bd.DA_ERR_WORKSPACE                       # no workspace
    # split partials: [splits, B, H, 2 streams, d_v] fp32 + (max, sum) per stream
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    assert lib.diffattn_v1_decode_workspace_size(2, 4, 256, 1024, 3) == \
        a256(3 * 2 * 4 * 2 * 256 * 4) + a256(3 * 2 * 4 * 2 * 2 * 4)
    assert lib.diffattn_v1_decode_num_splits(64, 16, 32768) >= 1
    assert lib.diffattn_v1_decode_num_splits(1, 1, 1000) == 1            # no split under 1024 keys


def test_v2_bwd_argument_checks(lib):
    p = bd.da_v2_bwd_params()
    p.B, p.N, p.h, p.h_kv, p.d, p.causal = 1, 256, 4, 2, 128, 1
    fake = 1 << 20
    for n in ("q", "o_heads", "dq"):
        setattr(p, n, bd.da_t4(fake, 1 << 18, 1 << 10, 128))
    for n in ("k", "v", "dk", "dv"):
        setattr(p, n, bd.da_t4(fake, 1 << 16, 1 << 8, 128))
    p.dout = bd.da_t4(fake, 1 << 17, 1 << 9, 128)
    p.lse, p.gate = fake, fake
    f = lib.diffattn_v2_bwd

    def with_(**kw):
        q = bd.da_v2_bwd_params.from_buffer_copy(p)
        for k, v in kw.items():
            setattr(q, k, v)
        return C.byref(q)
    assert f(with_(h_kv=3), None) == bd.DA_ERR_INVALID_ARG       # 2h not divisible into groups
    assert f(with_(h=1, h_kv=2), None) == bd.DA_ERR_INVALID_ARG  # a pair would straddle groups
    assert f(with_(d=96), None) == bd.DA_ERR_UNSUPPORTED
    assert f(with_(lse=None), None) == bd.DA_ERR_INVALID_ARG     # the forward's saves are needed
    assert f(with_(gate=None), None) == bd.DA_ERR_INVALID_ARG    # no gate and no x / w_lambda
    assert f(with_(dx=fake), None) == bd.DA_ERR_INVALID_ARG      # dX needs x and w_lambda
    assert f(with_(), None) == bd.DA_ERR_WORKSPACE
    assert f(with_(N=0), None) == bd.DA_OK                       # empty problem


def test_grouped_bwd_checks_and_workspace(lib):
    """Grouped backward: the forward's shape rules, its saves required, and at
    ratio 1 the same workspace as the V2 backward."""
    p = bd.da_grouped_bwd_params()
    p.B, p.N, p.h, p.ratio, p.h_kv, p.d, p.d_model, p.causal = 1, 256, 6, 3, 2, 128, 0, 1
    fake = 1 << 20
    for n in ("q", "k", "v", "o_heads", "dout", "dq", "dk", "dv"):
        setattr(p, n, bd.da_t4(fake, 256 * 8 * 128, 8 * 128, 128))
    p.gate = p.lse = fake
    f = lib.diffattn_grouped_bwd
    assert f(C.byref(p), None) == bd.DA_ERR_WORKSPACE  # valid shapes; no workspace
    bad = bd.da_grouped_bwd_params.from_buffer_copy(p)
    bad.h = 5  # not a multiple of the ratio
    assert f(C.byref(bad), None) == bd.DA_ERR_INVALID_ARG
    bad = bd.da_grouped_bwd_params.from_buffer_copy(p)
    bad.h_kv = 3  # 8 query heads do not split into 3 K/V groups
    assert f(C.byref(bad), None) == bd.DA_ERR_INVALID_ARG
    bad = bd.da_grouped_bwd_params.from_buffer_copy(p)
    bad.d = 96
    assert f(C.byref(bad), None) == bd.DA_ERR_UNSUPPORTED
    bad = bd.da_grouped_bwd_params.from_buffer_copy(p)
    bad.lse = None  # the forward's saves are required
    assert f(C.byref(bad), None) == bd.DA_ERR_INVALID_ARG
    bad = bd.da_grouped_bwd_params.from_buffer_copy(p)
    bad.gate = None  # the gate source: neither gate nor x and w_lambda
    assert f(C.byref(bad), None) == bd.DA_ERR_INVALID_ARG
    for B, N, h, dm in ((2, 8192, 32, 4096), (1, 300, 4, 0)):
        assert (lib.diffattn_grouped_bwd_workspace_size(B, N, h, 1, dm) ==
                lib.diffattn_v2_bwd_workspace_size(B, N, h, dm))
    assert lib.diffattn_grouped_bwd_workspace_size(2, 8192, 48, 3, 4096) > 0
    assert lib.diffattn_grouped_bwd_workspace_size(2, 8192, 47, 3, 4096) == 0
