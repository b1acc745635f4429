"""Seeded synthetic inputs for the drafter step, the draft block and greedy verification.

This module only draws random numbers and stores them; it performs no step of the drafter
arithmetic. Both the CUDA path and the CPU oracle are fed from it.

Recipe (one independent NumPy PCG64 stream per named tensor, keyed by (seed, name), so a
tensor's values do not depend on which other tensors were drawn or in what order):
  * matrices (projections, block weights, token_embd, centroids, the target's input
    embedding table): N(0, 0.02)
  * norm gains: 1 + N(0, 0.02), stored fp32
  * layer_scalar: U[0.5, 1]
  * token_ordering: a seeded permutation of 0..V-1 (int32)
  * shared K (one tensor per attention type) and the target's last hidden state: N(0, 1)
  * first token: uniform in [0, V); context length L_b fixed or U[lo, hi] (ragged);
    the constant position id is L_b
  * storage: bf16 by round-to-nearest-even for the bf16 shapes, fp32 for the fp32 shape;
    K padding beyond L_b is filled with NaN so that a read of it poisons the result.
The loop workload adds a synthetic target: base logits N(0,1) (bf16, clipped to [-8, 8]),
and per round, sequence and position an agreement bit ~ Bernoulli(p) and a uniform
alternative token; the target's row maximum (+16) is planted at the draft token when the
bit is set and at the alternative otherwise, so every row has a unique maximum.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
import zlib
from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np

from .configs import DrafterShape, Workload

BF16_NAN = np.uint16(0x7FC0)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, name: str, *extra: int) -> np.random.Generator:
    key = [int(seed), zlib.crc32(name.encode()) & 0xFFFFFFFF, *[int(e) for e in extra]]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def _normal(seed: int, name: str, shape, std: float, dtype: str, chunk_rows: int = 4096) -> np.ndarray:
    """N(0, std) in storage form: uint16 bf16 bits ("bf16") or float32 ("f32").

    Rows are drawn in chunks, each chunk from its own stream keyed by (seed, name, chunk),
    on a thread pool: the values do not depend on the number of threads.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16 if dtype == "bf16" else np.float32)
    flat = out.reshape(shape[0], -1) if len(shape) > 1 else out.reshape(1, -1)
    rows, cols = flat.shape

    def fill(ci: int) -> None:
        r0 = ci * chunk_rows
        r1 = min(rows, r0 + chunk_rows)
        v = _rng(seed, name, ci).standard_normal((r1 - r0, cols), dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        flat[r0:r1] = bf16_bits(v) if dtype == "bf16" else v

    n_chunks = (rows + chunk_rows - 1) // chunk_rows
    if n_chunks == 1 or rows * cols < (1 << 20):
        for ci in range(n_chunks):
            fill(ci)
    else:
        with _cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


def _gain(seed: int, name: str, n: int) -> np.ndarray:
    rng = _rng(seed, name)
    return (1.0 + 0.02 * rng.standard_normal(n)).astype(np.float32)


@dataclass
class Weights:
    """Drafter weights in storage form (bf16 bits as uint16, or float32) plus the target's
    input embedding table. Matrices are row-major [out][in]."""
    dtype: str
    pre_proj: np.ndarray        # [H][2*bb]
    post_proj: np.ndarray       # [bb][H]
    out_norm: np.ndarray        # [H] fp32
    token_embd: np.ndarray      # [V][H]
    centroids: Optional[np.ndarray]       # [C][H] or None (dense head)
    token_ordering: Optional[np.ndarray]  # [V] int32 or None
    target_embed: np.ndarray    # [V][bb]
    layers: List[Dict[str, object]]


def make_weights(shape: DrafterShape, seed: int) -> Weights:
    s, dt = shape, shape.dtype
    H, bb, V = s.hidden, s.backbone, s.vocab
    layers = []
    for i, lt in enumerate(s.layer_types):
        d = s.head_dim(lt)
        p = f"blk{i}."
        layers.append(dict(
            q=_normal(seed, p + "q", (s.n_head * d, H), 0.02, dt),
            q_norm=_gain(seed, p + "q_norm", d),
            o=_normal(seed, p + "o", (H, s.n_head * d), 0.02, dt),
            attn_norm=_gain(seed, p + "attn_norm", H),
            post_attn_norm=_gain(seed, p + "post_attn_norm", H),
            ffn_norm=_gain(seed, p + "ffn_norm", H),
            post_ffn_norm=_gain(seed, p + "post_ffn_norm", H),
            gate=_normal(seed, p + "gate", (s.ffn, H), 0.02, dt),
            up=_normal(seed, p + "up", (s.ffn, H), 0.02, dt),
            down=_normal(seed, p + "down", (H, s.ffn), 0.02, dt),
            layer_scalar=float(np.float32(_rng(seed, p + "layer_scalar").uniform(0.5, 1.0))),
        ))
    centroids = ordering = None
    if s.use_ordered_embeddings:
        centroids = _normal(seed, "centroids", (s.n_centroids, H), 0.02, dt)
        ordering = _rng(seed, "token_ordering").permutation(V).astype(np.int32)
    return Weights(
        dtype=dt,
        pre_proj=_normal(seed, "pre_proj", (H, 2 * bb), 0.02, dt),
        post_proj=_normal(seed, "post_proj", (bb, H), 0.02, dt),
        out_norm=_gain(seed, "out_norm", H),
        token_embd=_normal(seed, "token_embd", (V, H), 0.02, dt),
        centroids=centroids,
        token_ordering=ordering,
        target_embed=_normal(seed, "target_embed", (V, bb), 0.02, dt),
        layers=layers,
    )


@dataclass
class StepInputs:
    """Per-call inputs: hidden [B][bb], last_token [B], ctx_len [B], pos [B], and the shared K
    of each attention type, right-padded [B][Lmax][n_kv][d] with NaN beyond L_b."""
    hidden: np.ndarray
    last_token: np.ndarray
    ctx_len: np.ndarray
    pos: np.ndarray
    k_swa: Optional[np.ndarray]
    k_full: Optional[np.ndarray]


def make_ctx_len(workload: Workload, seed: int) -> np.ndarray:
    B = workload.batch
    if workload.ragged:
        return _rng(seed, "ctx_len").integers(workload.ctx_lo, workload.ctx + 1, size=B).astype(np.int32)
    return np.full(B, workload.ctx, dtype=np.int32)


def _kv(seed: int, name: str, B: int, Lmax: int, n_kv: int, d: int, ctx_len: np.ndarray, dt: str) -> np.ndarray:
    k = np.empty((B, Lmax, n_kv, d), dtype=np.uint16 if dt == "bf16" else np.float32)
    for b in range(B):
        L = int(ctx_len[b])
        k[b, :L] = _normal(seed, f"{name}.{b}", (L, n_kv, d), 1.0, dt)
        k[b, L:] = BF16_NAN if dt == "bf16" else np.float32(np.nan)
    return k


def make_step_inputs(shape: DrafterShape, workload: Workload, seed: int,
                     ctx_len: Optional[np.ndarray] = None) -> StepInputs:
    s, dt, B = shape, shape.dtype, workload.batch
    if ctx_len is None:
        ctx_len = make_ctx_len(workload, seed)
    ctx_len = np.asarray(ctx_len, dtype=np.int32)
    Lmax = int(workload.ctx)
    types = set(s.layer_types)
    k_swa = _kv(seed, "k_swa", B, Lmax, s.n_kv_head, s.head_dim_swa, ctx_len, dt) if "S" in types else None
    k_full = _kv(seed, "k_full", B, Lmax, s.n_kv_head, s.head_dim_full, ctx_len, dt) if "F" in types else None
    return StepInputs(
        hidden=_normal(seed, "hidden", (B, s.backbone), 1.0, dt),
        last_token=_rng(seed, "last_token").integers(0, s.vocab, size=B).astype(np.int32),
        ctx_len=ctx_len,
        pos=ctx_len.copy(),
        k_swa=k_swa,
        k_full=k_full,
    )


# ---------------------------------------------------------------------------------------
# Synthetic target for the draft+verify loop
# ---------------------------------------------------------------------------------------

PLANT_VALUE = 16.0


def base_target_logits(B: int, n_rows: int, V: int, seed: int) -> np.ndarray:
    """bf16 bits [B][n_rows][V], N(0,1) clipped to [-8, 8]."""
    rng = _rng(seed, "target_logits")
    out = np.empty((B, n_rows, V), dtype=np.uint16)
    for b in range(B):
        v = rng.standard_normal((n_rows, V), dtype=np.float32)
        np.clip(v, -8.0, 8.0, out=v)
        out[b] = bf16_bits(v)
    return out


def round_tables(B: int, n_draft: int, V: int, agree_p: float, seed: int, r: int):
    """Agreement bits [B][n_draft+1] (last row never agrees) and raw alternatives in
    [0, V-1) for round r."""
    rng = _rng(seed, "round", r)
    agree = rng.random((B, n_draft + 1)) < agree_p
    agree[:, n_draft] = False
    alt_raw = rng.integers(0, V - 1, size=(B, n_draft + 1)).astype(np.int64)
    return agree, alt_raw


def planted_targets(drafts: np.ndarray, agree: np.ndarray, alt_raw: np.ndarray, V: int) -> np.ndarray:
    """Token that holds the planted maximum of each target row [B][n+1].

    Row i < n: the draft token when agree[b,i], otherwise an alternative drawn uniformly
    from the V-1 tokens other than the draft. Row n (the bonus row): alt_raw itself.
    """
    drafts = np.asarray(drafts, dtype=np.int64)
    B, n = drafts.shape
    tgt = np.empty((B, n + 1), dtype=np.int64)
    alt = alt_raw[:, :n] + (alt_raw[:, :n] >= drafts)
    tgt[:, :n] = np.where(agree[:, :n], drafts, alt)
    tgt[:, n] = alt_raw[:, n]
    return tgt


def next_round_hidden(B: int, bb: int, seed: int, r: int, dtype: str = "bf16") -> np.ndarray:
    return _normal(seed, f"round_hidden.{r}", (B, bb), 1.0, dtype)
