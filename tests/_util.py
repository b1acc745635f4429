"""Test helpers: seeded inputs -> device tensors, and the comparison protocol between the
CUDA path and the oracle (tokens exact up to recorded near-ties, hidden states within
tolerance)."""
from __future__ import annotations

import functools
import math
from dataclasses import dataclass, field
from typing import List

import numpy as np
import torch

import oracle as O
from mtp_synth import configs as C
from mtp_synth import gen as G

# Tolerances of the precision contract: max-abs error of hidden states / logits.
TOL = {"bf16": 2e-2, "f32": 1e-4}
# A drafted token may differ from the oracle's only when the oracle's own margin at that
# step is below this: activations are fp32 in the kernels and fp64 in the oracle, so logits
# (|logit| ~ 1) differ by accumulation-order effects of ~1e-6; 1e-4 leaves a wide margin.
NEAR_TIE = {"bf16": 1e-4, "f32": 1e-4}


def to_torch(arr: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16" and arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def weights_to_device(w: G.Weights, device="cuda"):
    dt = w.dtype
    d = {
        "pre_proj": to_torch(w.pre_proj, dt, device), "post_proj": to_torch(w.post_proj, dt, device),
        "out_norm": to_torch(w.out_norm, "f32", device), "token_embd": to_torch(w.token_embd, dt, device),
        "centroids": None if w.centroids is None else to_torch(w.centroids, dt, device),
        "token_ordering": None if w.token_ordering is None else to_torch(w.token_ordering, "i32", device),
        "layers": [],
    }
    for L in w.layers:
        d["layers"].append({k: (v if k == "layer_scalar" else
                                to_torch(v, "f32" if k.endswith("norm") else dt, device)) for k, v in L.items()})
    return d, to_torch(w.target_embed, dt, device)


def inputs_to_device(inp: G.StepInputs, dtype: str, device="cuda"):
    return dict(
        hidden=to_torch(inp.hidden, dtype, device),
        last_token=to_torch(inp.last_token, "i32", device),
        ctx_len=to_torch(inp.ctx_len, "i32", device),
        pos=to_torch(inp.pos, "i32", device),
        k_swa=None if inp.k_swa is None else to_torch(inp.k_swa, dtype, device),
        k_full=None if inp.k_full is None else to_torch(inp.k_full, dtype, device),
    )


@functools.lru_cache(maxsize=4)
def config_data(index: int, batch: int = 0, ctx: int = 0):
    """Seeded weights and step inputs of a benchmark configuration (optionally with a
    different batch / context for smaller cases)."""
    cfg = C.config(index)
    wl = cfg.workload
    if batch or ctx:
        from dataclasses import replace
        wl = replace(wl, batch=batch or wl.batch, ctx=ctx or wl.ctx,
                     ctx_lo=None if wl.ctx_lo is None else min(wl.ctx_lo, ctx or wl.ctx))
    w = G.make_weights(cfg.shape, wl.seed)
    inp = G.make_step_inputs(cfg.shape, wl, wl.seed)
    return cfg.shape, wl, w, inp


@functools.lru_cache(maxsize=4)
def decoded(index: int, batch: int = 0, ctx: int = 0):
    shape, wl, w, inp = config_data(index, batch, ctx)
    return O.Shape.of(shape), O.decode_weights(w)


@dataclass
class Comparison:
    steps_compared: int = 0
    tie_divergences: List[tuple] = field(default_factory=list)
    max_hidden_err: float = 0.0


def compare_block(gpu_tokens: np.ndarray, gpu_hidden, ref: O.BlockResult, dtype: str) -> Comparison:
    """Tokens must match exactly, hidden states within TOL. A token may differ only at a
    step where the oracle itself has a near-tie (top-2 logit gap, or the k-th / (k+1)-th
    centroid gap, below NEAR_TIE); later steps of that sequence are then not compared,
    since the two paths continue from different tokens."""
    out = Comparison()
    B, n = ref.tokens.shape
    tol, delta = TOL[dtype], NEAR_TIE[dtype]
    for b in range(B):
        for i in range(n):
            if gpu_hidden is not None:
                err = float(np.max(np.abs(gpu_hidden[b, i].astype(np.float64) - ref.hidden_out[b, i])))
                out.max_hidden_err = max(out.max_hidden_err, err)
                assert err <= tol, f"hidden state of sequence {b} step {i}: max-abs error {err} > {tol}"
            out.steps_compared += 1
            if int(gpu_tokens[b, i]) != int(ref.tokens[b, i]):
                gap = min(ref.logit_gap[b, i], ref.kth_gap[b, i])
                assert gap < delta, (f"token mismatch at sequence {b} step {i}: gpu {gpu_tokens[b, i]} oracle "
                                     f"{ref.tokens[b, i]} with oracle margin {gap} >= {delta}")
                out.tie_divergences.append((b, i, gap))
                break
    return out


def oracle_block(index: int, n_draft=None, batch: int = 0, ctx: int = 0, **kw) -> O.BlockResult:
    shape, wl, w, inp = config_data(index, batch, ctx)
    s, W = decoded(index, batch, ctx)
    return O.draft_block(s, W, inp.hidden, inp.last_token, inp.k_swa, inp.k_full, inp.ctx_len, inp.pos,
                         n_draft or wl.n_draft, **kw)


def expected_accept(p: float, n: int):
    mean = sum(p ** i for i in range(1, n + 1))
    var = sum((2 * i - 1) * p ** i for i in range(1, n + 1)) - mean ** 2
    return mean, math.sqrt(var)
