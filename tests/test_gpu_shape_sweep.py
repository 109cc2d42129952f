"""A seeded sweep of drawn shapes through every entry point against the fp64
oracle, with the bars of the fixed-shape parity tests (their checks are
reused as they are): batch, length (one token, under a tile, whole tiles,
ragged tails over several tiles), head counts and group sizes, head dims,
causal or not, the layer index, an RMSNorm weight, decode lengths and split
counts, the softmax scale, the V1 RMSNorm epsilon, the V1 backward's
deterministic mode and strided input views are drawn together, so that combinations the hand-picked cases leave
out are run as well.  The draws are fixed by the seed; the CPU test checks
that every drawn shape is one the entry points accept and that the sweep
spans the categories it claims."""

import random

import numpy as np
import pytest
import torch

SEED = 7309
CASES = 12

# length categories, cycled over a sweep's cases: under one 128-row tile,
# whole tiles, ragged over several tiles
def _length(rng, i, cap):
    kind = i % 3
    if kind == 0:
        return rng.choice([1, rng.randint(2, 127)])
    if kind == 1:
        return 128 * rng.randint(1, cap // 128)
    return 128 * rng.randint(1, cap // 128 - 1) + rng.randint(1, 127)


def _eps(rng):
    """The V1 RMSNorm epsilon: mostly the default, sometimes large enough
    (against mean O^2 of about 0.05) to change the result visibly."""
    return float(np.float32(rng.choice([1e-5, 1e-5, 1e-3, 3e-2])))


def sweep_cases(op, n=CASES, seed=SEED):
    rng = random.Random(f"{op}/{seed}")
    cases = []
    for i in range(n):
        causal = i % 2 == 0 or rng.random() < 0.5
        # every third case a softmax scale other than the default 1/sqrt(d),
        # exactly representable in fp32 as the interface takes it
        scale = float(np.float32(rng.uniform(0.03, 0.2))) if i % 3 == 2 else None
        if op in ("v1_fwd", "v1_bwd"):
            dqk, dv = rng.choice([(128, 256), (64, 128)])
            cap = 700 if op == "v1_fwd" else 400
            cases.append(dict(B=rng.randint(1, 3), N=_length(rng, i, cap), H=rng.randint(1, 3 if op == "v1_bwd" else 4),
                              dqk=dqk, dv=dv, causal=causal, layer=rng.randint(1, 28),
                              weighted=rng.random() < 0.3, eps=_eps(rng)))
            if op == "v1_bwd":  # every fourth step with dQ through the ordered slots
                cases[-1]["det"] = i % 4 == 1
        elif op == "v1_fwd_f32":
            # the fp32 path: any d_qk <= 128, d_v <= 256 with d_v % 32 == 0
            cases.append(dict(B=rng.randint(1, 3), N=_length(rng, i, 384), H=rng.randint(1, 4),
                              dqk=rng.randint(1, 128), dv=32 * rng.randint(1, 8), causal=causal,
                              layer=rng.randint(1, 28), weighted=rng.random() < 0.3, eps=_eps(rng)))
        elif op in ("v2_fwd", "v2_bwd"):
            hkv = rng.choice([1, 2, 4])
            per = rng.choice([1, 2] if op == "v2_bwd" else [1, 2, 4])  # head pairs per K/V head
            cap = 700 if op == "v2_fwd" else 400
            cases.append(dict(B=rng.randint(1, 3), N=_length(rng, i, cap), h=hkv * per, hkv=hkv,
                              d=rng.choice([64, 128]), dm=rng.choice([64, 128, 192, 256]), causal=causal))
        elif op in ("grouped_fwd", "grouped_bwd"):
            ratio = rng.choice([2, 3, 4])
            hkv = rng.choice([1, 2])
            # query heads per K/V head, (ratio + 1) * groups per K/V head,
            # must be even
            groups = hkv * (rng.choice([1, 2]) if ratio % 2 else 2)
            cap = 600 if op == "grouped_fwd" else 300
            cases.append(dict(B=rng.randint(1, 2), N=_length(rng, i, cap), h=groups * ratio, ratio=ratio, hkv=hkv,
                              d=rng.choice([64, 128]), dm=rng.choice([128, 256]), causal=causal))
        elif op == "v2_decode":
            hkv = rng.choice([1, 2, 8])
            B = rng.randint(1, 4)
            L = rng.randint(1, 3000)
            seqlens = [L] + [rng.randint(1, L) for _ in range(B - 1)]
            cases.append(dict(B=B, L=L, h=hkv * rng.choice([1, 2, 4]), hkv=hkv, d=rng.choice([64, 128]),
                              dm=rng.choice([64, 256]), seqlens=seqlens, splits=rng.choice([0, 1, 2, 3, 5])))
        elif op == "v1_decode":
            B = rng.randint(1, 4)
            L = rng.randint(1, 3000)
            seqlens = [L] + [rng.randint(1, L) for _ in range(B - 1)]
            dqk, dv = rng.choice([(128, 256), (64, 128)])
            cases.append(dict(B=B, L=L, H=rng.randint(1, 4), dqk=dqk, dv=dv, seqlens=seqlens,
                              splits=rng.choice([0, 1, 2, 3, 5]), layer=rng.randint(1, 28),
                              weighted=rng.random() < 0.3, eps=_eps(rng)))
        else:
            raise ValueError(op)
        cases[-1]["scale"] = scale
        # every fourth case reads its 4-D inputs through strided views
        cases[-1]["strided"] = i % 4 == 3
    return cases


OPS = ("v1_fwd", "v1_bwd", "v1_fwd_f32", "v2_fwd", "v2_bwd", "grouped_fwd", "grouped_bwd", "v2_decode",
       "v1_decode")


def _ids(op):
    return [f"{op}-{i}" for i in range(CASES)]


def test_sweep_shapes_are_valid():
    """Every drawn shape satisfies the entry points' documented constraints,
    and each sweep spans short, whole-tile and ragged lengths (decode:
    several lengths and split counts)."""
    for op in OPS:
        cases = sweep_cases(op)
        assert len(cases) == CASES
        assert sweep_cases(op) == cases  # fixed by the seed
        for c in cases:
            if op.startswith("v2") and op != "v2_decode":
                assert c["h"] % c["hkv"] == 0 and c["dm"] % 64 == 0 and c["d"] in (64, 128)
            if op.startswith("grouped"):
                groups = c["h"] // c["ratio"]
                assert c["h"] % c["ratio"] == 0 and groups % c["hkv"] == 0
                G = groups * (c["ratio"] + 1) // c["hkv"]  # query heads per K/V head
                assert G % (c["ratio"] + 1) == 0 and G % 2 == 0
            if op.endswith("decode"):
                assert len(c["seqlens"]) == c["B"] and max(c["seqlens"]) == c["L"]
                assert all(1 <= s <= c["L"] for s in c["seqlens"])
            if op == "v2_decode":
                assert c["h"] % c["hkv"] == 0
            if op in ("v1_fwd", "v1_bwd"):
                assert (c["dqk"], c["dv"]) in ((128, 256), (64, 128))
            if op == "v1_fwd_f32":
                assert 1 <= c["dqk"] <= 128 and c["dv"] <= 256 and c["dv"] % 32 == 0
            assert c["scale"] is None or (0 < c["scale"] < 1 and float(np.float32(c["scale"])) == c["scale"])
        assert any(c["scale"] is not None for c in cases) and any(c["scale"] is None for c in cases)
        if op.startswith("v1"):
            assert any(c["eps"] > 1e-4 for c in cases) and all(c["eps"] > 0 for c in cases)
        if op == "v1_bwd":
            assert any(c["det"] for c in cases) and not all(c["det"] for c in cases)
        if not op.endswith("decode"):
            ns = [c["N"] for c in cases]
            assert any(n < 128 for n in ns) and any(n % 128 == 0 for n in ns)
            assert any(n > 128 and n % 128 for n in ns)
            assert any(c["causal"] for c in cases)


def test_strided_views_hold_the_values_and_nan_around_them():
    """The strided-view helper (CPU tensors here): each view equals its source,
    its batch, row and head strides differ from a contiguous tensor's, it
    starts 16-byte aligned with strides in whole 16-byte steps (what the
    interface requires of bf16 tensors), and everything of its buffer outside
    the view is NaN."""
    g = torch.Generator().manual_seed(3)
    t = {"a": torch.randn((2, 37, 3, 64), generator=g).to(torch.bfloat16),
         "b": torch.randn((1, 5, 2, 128), generator=g).to(torch.bfloat16)}
    for seed in range(20):
        out = _strided(t, ("a", "b"), seed)
        for n, x in t.items():
            v = out[n]
            assert torch.equal(v, x)
            assert v.stride(3) == 1 and v.stride()[:3] != x.contiguous().stride()[:3]
            assert v.data_ptr() % 16 == 0 and all((st * 2) % 16 == 0 for st in v.stride()[:3])
            base = v.storage_offset()
            buf = torch.empty(0, dtype=v.dtype).set_(v.untyped_storage())
            mask = torch.ones(buf.numel(), dtype=torch.bool)
            idx = torch.arange(v.numel()).view(v.shape)
            flat = (base + sum(idx.new_tensor(list(range(sz))).view([-1 if i == d else 1 for i in range(4)]) * st
                               for d, (sz, st) in enumerate(zip(v.shape, v.stride())))).reshape(-1)
            mask[flat] = False
            assert torch.isnan(buf[mask].float()).all()


# ------------------------------------------------------------------- GPU ----

@pytest.fixture
def gpu_ops():
    """The binding and the fixed-shape tests' checks; afterwards the device
    status word must be clean."""
    import test_gpu_grouped as tg
    import test_gpu_grouped_bwd as tgb
    import test_gpu_small as tsm
    import test_gpu_v1 as tv1
    import test_gpu_v1_bwd as tv1b
    import test_gpu_v1_decode as tv1d
    import test_gpu_v2 as tv2
    import test_gpu_v2_bwd as tv2b
    from differential_attention_diff_gb300 import binding as bd
    ns = dict(bd=bd, tg=tg, tgb=tgb, tsm=tsm, tv1=tv1, tv1b=tv1b, tv1d=tv1d, tv2=tv2, tv2b=tv2b)
    yield ns
    assert bd.diffattn_get_device_status() == bd.DA_OK


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _ss(c):
    return 0.0 if c["scale"] is None else c["scale"]


def _strided(t, names, seed):
    """The 4-D tensors `names` of t as views into larger NaN-filled buffers:
    one or two extra heads and a few extra rows per batch, the view starting
    at a drawn head and row offset, so that every batch, row and head stride
    differs from the contiguous one.  A kernel that read outside its view
    would pick up NaN and fail parity."""
    rng = random.Random(seed)
    out = dict(t)
    for n in names:
        x = t[n]
        B, N, H, D = x.shape
        ph, pn = rng.randint(1, 2), rng.randint(1, 5)
        oh, on = rng.randint(0, ph), rng.randint(0, pn)
        buf = torch.full((B, N + pn, H + ph, D), float("nan"), dtype=x.dtype, device=x.device)
        v = buf[:, on:on + N, oh:oh + H]
        v.copy_(x)
        out[n] = v
    return out


def _rms_weight(n, seed):
    return 0.5 + torch.rand(n, generator=torch.Generator().manual_seed(seed), dtype=torch.float32).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v1_fwd"), ids=_ids("v1_fwd"))
def test_sweep_v1_fwd(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    bd, tv1 = gpu_ops["bd"], gpu_ops["tv1"]
    t = synth.v1_inputs(c["B"], c["N"], c["H"], c["dqk"], c["dv"], "bf16", seed=11000 + c["N"], device="cuda")
    if c["strided"]:
        t = _strided(t, ("q1", "q2", "k1", "k2", "v"), 11002 + c["N"])
    li = bd.diffattn_lambda_init(c["layer"])
    w = _rms_weight(c["dv"], 11001) if c["weighted"] else None
    y, sv = bd.diffattn_v1_fwd(*(t[n] for n in tv1.NAMES), li, save=True, causal=c["causal"], rms_weight=w,
                               softmax_scale=_ss(c), rms_eps=c["eps"])
    torch.cuda.synchronize()
    tv1._check(t, li, y, sv, causal=c["causal"], w=w, scale=c["scale"], eps=c["eps"])


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v1_bwd"), ids=_ids("v1_bwd"))
def test_sweep_v1_bwd(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    from oracle import diffattn_oracle as orc
    bd, tv1b = gpu_ops["bd"], gpu_ops["tv1b"]
    t = synth.v1_inputs(c["B"], c["N"], c["H"], c["dqk"], c["dv"], "bf16", seed=12000 + c["N"], device="cuda",
                        with_dy=True)
    if c["strided"]:
        t = _strided(t, ("q1", "q2", "k1", "k2", "v", "dy"), 12002 + c["N"])
    li = float(np.float32(bd.diffattn_lambda_init(c["layer"])))
    w = _rms_weight(c["dv"], 12001) if c["weighted"] else None
    wf = None if w is None else _f64(w)
    sc, eps = c["scale"], c["eps"]
    ref = orc.v1_backward(*(_f64(t[n]) for n in tv1b.NAMES), li, _f64(t["dy"]), causal=c["causal"], rms_weight=wf,
                          scale=sc, eps=eps)
    tv1b._compare(tv1b._run_exact_saves(t, li, causal=c["causal"], w=w, scale=sc, eps=eps), ref,
                  tv1b._model(t, li, causal=c["causal"], w=w, scale=sc, eps=eps), bar="bwd", layer=c["layer"])
    tv1b._compare(tv1b._run(t, li, causal=c["causal"], w=w, scale=sc, eps=eps, deterministic=c["det"]), ref,
                  tv1b._model(t, li, causal=c["causal"], w=w, step=True, scale=sc, eps=eps), bar="step",
                  layer=c["layer"])


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v2_fwd"), ids=_ids("v2_fwd"))
def test_sweep_v2_fwd(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    from oracle import diffattn_oracle as orc
    bd, tv2 = gpu_ops["bd"], gpu_ops["tv2"]
    t = synth.v2_inputs(c["B"], c["N"], c["h"], c["hkv"], c["d"], c["dm"], seed=13000 + c["N"], device="cuda")
    if c["strided"]:
        t = _strided(t, ("q", "k", "v"), 13002 + c["N"])
    lse = torch.empty((c["B"], 2 * c["h"], c["N"]), dtype=torch.float32, device="cuda")
    out = bd.diffattn_v2_fwd(t["q"], t["k"], t["v"], x=t["x"], w_lambda=t["w_lambda"], lse=lse, causal=c["causal"],
                             softmax_scale=_ss(c))
    torch.cuda.synchronize()
    gate = orc.v2_gate(_f64(t["x"]), _f64(t["w_lambda"]))
    tv2._check_pairs(t, out, gate, lse=lse, causal=c["causal"], scale=c["scale"])


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v2_bwd"), ids=_ids("v2_bwd"))
def test_sweep_v2_bwd(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    tv2b = gpu_ops["tv2b"]
    t = synth.v2_inputs(c["B"], c["N"], c["h"], c["hkv"], c["d"], c["dm"], seed=14000 + c["N"], device="cuda",
                        with_dout=True)
    if c["strided"]:
        t = _strided(t, ("q", "k", "v", "dout"), 14002 + c["N"])
    sc = c["scale"]
    ref, fwd, model = tv2b._reference(t, causal=c["causal"], scale=sc)
    tv2b._compare(tv2b._run_exact_saves(t, fwd, causal=c["causal"], scale=sc), ref, model, bar="bwd")
    tv2b._compare(tv2b._run(t, causal=c["causal"], scale=sc), ref, model, bar="step")


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("grouped_fwd"), ids=_ids("grouped_fwd"))
def test_sweep_grouped_fwd(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    bd, tg = gpu_ops["bd"], gpu_ops["tg"]
    t = synth.grouped_inputs(c["B"], c["N"], c["h"], c["ratio"], c["hkv"], c["d"], c["dm"], seed=15000 + c["N"],
                             device="cuda")
    if c["strided"]:
        t = _strided(t, ("q", "k", "v"), 15002 + c["N"])
    out = bd.diffattn_grouped_fwd(t["q"], t["k"], t["v"], c["ratio"], x=t["x"], w_lambda=t["w_lambda"],
                                  causal=c["causal"], softmax_scale=_ss(c))
    torch.cuda.synchronize()
    tg._check(t, c["ratio"], out, causal=c["causal"], scale=c["scale"])


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("grouped_bwd"), ids=_ids("grouped_bwd"))
def test_sweep_grouped_bwd(c, gpu_ops):
    tgb = gpu_ops["tgb"]
    t = tgb._inputs(c["B"], c["N"], c["h"], c["ratio"], c["hkv"], c["d"], c["dm"], seed=16000 + c["N"])
    if c["strided"]:
        t = _strided(t, ("q", "k", "v", "dout"), 16002 + c["N"])
    sc = c["scale"]
    ref, model = tgb._reference(t, c["ratio"], causal=c["causal"], scale=sc)
    tgb._compare(tgb._run_exact_saves(t, c["ratio"], ref, causal=c["causal"], scale=sc), ref, model, bar="bwd")
    tgb._compare(tgb._run(t, c["ratio"], causal=c["causal"], scale=sc), ref, model, bar="step")


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v2_decode"), ids=_ids("v2_decode"))
def test_sweep_v2_decode(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    bd, tsm = gpu_ops["bd"], gpu_ops["tsm"]
    t = synth.decode_inputs(c["B"], c["L"], c["h"], c["hkv"], c["d"], c["dm"], seed=17000 + c["L"], device="cuda",
                            seqlens=c["seqlens"])
    if c["strided"]:
        t = _strided(t, ("k_cache", "v_cache"), 17002 + c["L"])
    out = bd.diffattn_v2_decode(t["q"], t["k_cache"], t["v_cache"], seqlens=t["seqlens"], x=t["x"],
                                w_lambda=t["w_lambda"], num_splits=c["splits"], softmax_scale=_ss(c))
    torch.cuda.synchronize()
    tsm._decode_check(t, out, scale=c["scale"])


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v1_decode"), ids=_ids("v1_decode"))
def test_sweep_v1_decode(c, gpu_ops):
    from differential_attention_diff_gb300 import synth
    bd, tv1d = gpu_ops["bd"], gpu_ops["tv1d"]
    t = synth.v1_decode_inputs(c["B"], c["L"], c["H"], c["dqk"], c["dv"], seed=18000 + c["L"], device="cuda",
                               seqlens=c["seqlens"])
    if c["strided"]:
        t = _strided(t, ("k1_cache", "k2_cache", "v_cache"), 18002 + c["L"])
    li = bd.diffattn_lambda_init(c["layer"])
    w = _rms_weight(c["dv"], 18001) if c["weighted"] else None
    tv1d._check(t, li, tv1d._run(t, li, num_splits=c["splits"], rms_weight=w, softmax_scale=_ss(c),
                                 rms_eps=c["eps"]), w=w, scale=c["scale"], eps=c["eps"])


@pytest.mark.gpu
@pytest.mark.parametrize("c", sweep_cases("v1_fwd_f32"), ids=_ids("v1_fwd_f32"))
def test_sweep_v1_fwd_f32(c, gpu_ops):
    """The fp32 V1 path (its own SIMT kernel) at drawn head dims: Y and O2
    within 1e-4 * RMS(V), the LSEs within 1e-4, rstd within 1e-4 relative."""
    from differential_attention_diff_gb300 import synth
    from oracle import diffattn_oracle as orc
    bd, tsm = gpu_ops["bd"], gpu_ops["tsm"]
    names = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
    t = synth.v1_inputs(c["B"], c["N"], c["H"], c["dqk"], c["dv"], dtype="f32", seed=19000 + c["N"], device="cuda")
    li = bd.diffattn_lambda_init(c["layer"])
    w = _rms_weight(c["dv"], 19001) if c["weighted"] else None
    out, sv = bd.diffattn_v1_fwd(*(t[n] for n in names), li, save=True, causal=c["causal"], rms_weight=w,
                                 softmax_scale=_ss(c), rms_eps=c["eps"])
    torch.cuda.synchronize()
    ref = orc.v1_forward(*(_f64(t[n]) for n in names), float(np.float32(li)), causal=c["causal"],
                         rms_weight=None if w is None else _f64(w), scale=c["scale"], eps=c["eps"])
    tol = tsm.F32_TOL * float(np.sqrt(np.mean(_f64(t["v"]) ** 2)))
    worst = max(tsm.maxdiff(_f64(out), ref["y"]), tsm.maxdiff(_f64(sv["o2"]), ref["o2"])) / tol
    tsm.record({"y_o2": worst})
    assert worst <= 1.0, worst
    assert tsm.maxdiff(_f64(sv["lse1"]), ref["lse1"]) <= 1e-4
    assert tsm.maxdiff(_f64(sv["lse2"]), ref["lse2"]) <= 1e-4
    assert np.max(np.abs(_f64(sv["rstd"]) / ref["rstd"] - 1)) <= 1e-4
