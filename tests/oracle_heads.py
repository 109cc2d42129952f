"""The fp64 oracle (and the bf16 rounding model) of the V1 backward, one head
per task, spread over a process pool (test infrastructure).

At the training-step workload's full size (B1 H16 N8192) the oracle's
backward of one head forms several 8192 x 8192 fp64 matrices; heads are
independent, so the sixteen heads run as separate tasks in a pool started
with the "spawn" method (a pool forked from a process that has used the GPU
can hang).  Nothing here adds arithmetic: each task calls
``oracle.diffattn_oracle.v1_backward`` / ``v1_forward`` and
``bf16_model.rounded_backward`` on one head's arrays, and the caller stacks
the heads.  The four lambda-vector gradients are linear in dlambda, which
sums over heads, so the whole problem's lambda-vector gradients are the sums
of the per-head ones.
"""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

NAMES = ("q1", "q2", "k1", "k2", "v", "lq1", "lk1", "lq2", "lk2")
HEAD_GRADS = ("dq1", "dq2", "dk1", "dk2", "dv")
LAM_GRADS = ("dlq1", "dlk1", "dlq2", "dlk2")


def _one_head(task):
    from bf16_model import rounded_backward, rounded_forward
    from oracle import diffattn_oracle as orc

    f, li, causal, step = task
    ref = orc.v1_backward(*(f[n] for n in NAMES), li, f["dy"], causal=causal)
    fwd = orc.v1_forward(*(f[n] for n in NAMES), li, causal=causal)
    if step:
        model = rounded_backward(f, rounded_forward(f, fwd, li, causal=causal), li, causal=causal, exact_fwd=fwd)
    else:
        model = rounded_backward(f, fwd, li, causal=causal)
    keep = HEAD_GRADS + LAM_GRADS + ("dlam",)
    return {n: ref[n] for n in keep}, {n: model[n] for n in HEAD_GRADS + ("dlam", "dlam_ss") if n in model}


def v1_backward_by_head(f, li, causal=True, workers=None, step=False):
    """f: fp64 arrays of the V1 inputs and dy ([B, N, H, D]; lambda vectors
    [d_qk]).  Returns (ref, model) for every head, in the layout of
    ``orc.v1_backward`` / ``rounded_backward`` on the whole problem; with
    step=True the model also rounds the forward's storage points
    (``rounded_forward``), as for the training step."""
    B, N, H, _ = f["q1"].shape
    tasks = []
    for b in range(B):
        for h in range(H):
            fh = {n: (f[n][b:b + 1, :, h:h + 1] if f[n].ndim == 4 else f[n]) for n in NAMES + ("dy",)}
            tasks.append((fh, li, causal, step))
    if workers is None:
        workers = max(1, min(len(tasks), (os.cpu_count() or 4) // 4))
    if workers == 1:
        results = [_one_head(t) for t in tasks]
    else:
        with mp.get_context("spawn").Pool(workers) as pool:
            results = pool.map(_one_head, tasks, chunksize=1)
    ref = {n: np.zeros_like(f["v" if n == "dv" else "q1"]) for n in HEAD_GRADS}
    model = {n: np.zeros_like(ref[n]) for n in HEAD_GRADS}
    for n in LAM_GRADS:
        ref[n] = np.zeros_like(f["lq1"])
    ref["dlam"] = model["dlam"] = 0.0
    for i, (r, m) in enumerate(results):
        b, h = divmod(i, H)
        for n in HEAD_GRADS:
            ref[n][b, :, h] = r[n][0, :, 0]
            model[n][b, :, h] = m[n][0, :, 0]
        for n in LAM_GRADS:
            ref[n] += r[n]
        ref["dlam"] += r["dlam"]
        model["dlam"] += m["dlam"]
        if "dlam_ss" in m:  # heads' rows add their squared errors
            model["dlam_ss"] = model.get("dlam_ss", 0.0) + m["dlam_ss"]
    return ref, model
