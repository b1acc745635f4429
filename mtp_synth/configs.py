"""Drafter shapes and workloads of the five benchmark configurations.

Pure data: sizes, layer schedules and workload parameters. Nothing here computes any part
of the drafter step; both the CUDA path and the CPU oracle receive the same tensors built
from these descriptions by ``mtp_synth.gen``.

Shapes follow the published variants of the Gemma-4 assistant drafter:
  * "Gemma 4 Multi-Token Prediction (MTP) drafter" (llama.cpp gemma4-assistant doc),
    sections "Tensor schema" and "Variants supported": hidden 256, 4 blocks, backbone
    1536 (E2B) / 2560 (E4B), 2048 centroids, top-32, vocabulary 262144.
  * "Gemma 4 Assistant tensor inventory", section "HF config highlights": three sliding
    layers plus one full layer, attention_k_eq_v, backbone 2816 and a dense tied head
    for the 26B-A4B drafter.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional, Tuple


@dataclass(frozen=True)
class DrafterShape:
    name: str
    dtype: str                  # "bf16" (matrices, KV, embeddings stored bf16) or "f32"
    backbone: int               # target hidden size (bb)
    hidden: int                 # assistant hidden size (H)
    layer_types: Tuple[str, ...]  # "S" sliding / "F" full, one per block
    n_head: int
    head_dim_swa: int
    head_dim_full: int
    n_kv_head: int
    ffn: int
    vocab: int
    n_centroids: int
    top_k: int
    window: int
    use_ordered_embeddings: bool
    rms_eps: float = 1e-6
    attn_scale: float = 0.0     # 0 -> 1/sqrt(head_dim)
    rope_theta_swa: float = 1.0e4
    rope_theta_full: float = 1.0e6

    @property
    def n_layers(self) -> int:
        return len(self.layer_types)

    def head_dim(self, layer_type: str) -> int:
        return self.head_dim_full if layer_type == "F" else self.head_dim_swa

    @property
    def vsc(self) -> int:
        """Vocabulary entries per centroid (vocab / n_centroids)."""
        return self.vocab // self.n_centroids if self.n_centroids else 0


@dataclass(frozen=True)
class Workload:
    batch: int
    ctx: int                          # fixed context length, or the upper bound when ragged
    ctx_lo: Optional[int] = None      # ragged: L_b ~ U[ctx_lo, ctx] (inclusive)
    n_draft: int = 1
    rounds: int = 1                   # draft+verify rounds (the loop workload)
    agree_p: float = 0.0              # per-position agreement probability of the synthetic target
    seed: int = 1000

    @property
    def ragged(self) -> bool:
        return self.ctx_lo is not None


@dataclass(frozen=True)
class Config:
    index: int
    label: str
    shape: DrafterShape
    workload: Workload
    description: str = field(default="", compare=False)


TINY_F32 = DrafterShape(
    name="tiny-f32", dtype="f32", backbone=128, hidden=64, layer_types=("F",), n_head=2,
    head_dim_swa=32, head_dim_full=32, n_kv_head=1, ffn=256, vocab=4096, n_centroids=64,
    top_k=4, window=0, use_ordered_embeddings=True)

E2B = DrafterShape(
    name="e2b", dtype="bf16", backbone=1536, hidden=256, layer_types=("S", "S", "S", "F"),
    n_head=4, head_dim_swa=256, head_dim_full=512, n_kv_head=1, ffn=2048, vocab=262144,
    n_centroids=2048, top_k=32, window=512, use_ordered_embeddings=True)

E4B = replace(E2B, name="e4b", backbone=2560)

# E4B with the two shared KV heads one page lists (the benchmark workload follows the other
# page's "same head structure as E2B", one KV head); a parity-test shape only.
E4B_KV2 = replace(E4B, name="e4b-kv2", n_kv_head=2)

A4B_DENSE = DrafterShape(
    name="26b-a4b-dense", dtype="bf16", backbone=2816, hidden=1024,
    layer_types=("S", "S", "S", "F"), n_head=8, head_dim_swa=128, head_dim_full=128,
    n_kv_head=2, ffn=4096, vocab=262144, n_centroids=0, top_k=0, window=1024,
    use_ordered_embeddings=False)

CONFIGS = (
    Config(0, "tiny fp32 single step", TINY_F32,
           Workload(batch=1, ctx=64, n_draft=1, seed=1000)),
    Config(1, "E2B bf16 B=1 ctx 4096 block 4", E2B,
           Workload(batch=1, ctx=4096, n_draft=4, seed=1001)),
    Config(2, "E4B bf16 B=8 ragged ctx [4096,32768] block 6", E4B,
           Workload(batch=8, ctx=32768, ctx_lo=4096, n_draft=6, seed=1002)),
    Config(3, "26B-A4B-shape dense head B=32 ctx 8192 block 4", A4B_DENSE,
           Workload(batch=32, ctx=8192, n_draft=4, seed=1003)),
    Config(4, "E2B draft+verify B=64 ctx 2048 block 8 x1000 rounds", E2B,
           Workload(batch=64, ctx=2048, n_draft=8, rounds=1000, agree_p=0.6, seed=1004)),
)


def config(i: int) -> Config:
    return CONFIGS[i]
